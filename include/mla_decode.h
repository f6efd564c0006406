/*
 * mla_decode.h -- C ABI of the GB300 (sm_103a) MLA latent-decode library.
 *
 * The library computes weight-absorbed multi-head latent attention (MLA)
 * decode with MTP verification over a paged latent KV cache, as split-KV
 * flash-decoding: a partial (O, LSE) per KV split (and per context shard),
 * merged by LSE, either as two launches (mla_decode_partial, mla_lse_combine)
 * or fused into one (mla_decode).
 *
 * Pages that define the operations (cited by title and section):
 *   [VRAM-KV]  "Resident VRAM: weights and KV cache" (zdszero.github.io),
 *              section "KV 账：每 token 字节由注意力架构决定" (KV ledger): the MLA
 *              cache stores one latent row per token of kv_lora_rank (512,
 *              c_kv) + qk_rope_head_dim (64, RoPE key) elements, no head dim.
 *   [VRAM-POOL] same page, sections "cell_size：每 token 字节的代码形态" and
 *              "req_to_token 的大小从哪来": the per-layer pool is
 *              (size + page_size, 1, 576); req_to_token is an int32 2-D table
 *              [requests, context] from token index to pool slot.
 *   [K3-MLA]   "Kimi K3 decode on 2x8 B200: DP16 vs DP2 x DCP8"
 *              (zdszero.github.io), section "MLA：字节守恒，但 DP16 的 kernel 被
 *              wave 量化拖慢" (MLA: bytes conserved, the DP16 kernel is slowed
 *              by wave quantisation): the decode kernel's split count and grid,
 *              the partial (O, LSE) exchange and the LSE combine
 *              (dcp_lse_combine), 96 heads with replicated Q on every shard.
 *   [K3-SPLIT] same page, section "问题：同样 16 张卡、同样的并发，按什么切": the
 *              latent KV split token-interleaved, slot p on shard p % 8.
 *   [K3-INTRO] same page, opening paragraphs: 5 tokens verified per request
 *              per step (q_len = 5, causal among the draft tokens).
 *   [K3-MEM]   same page, section "显存：固定开销决定状态池有多大": 96 heads, qk
 *              head dim 192 (128 nope + 64 rope), absorbed query 512-d.
 *
 * Conventions for every entry point:
 *   - Device pointers are CUDA device memory owned by the caller; host
 *     pointers are marked "host".  The library allocates nothing and never
 *     frees caller memory.  It keeps no state between calls, except the
 *     static scratch of mla_decode_scratch (whose counters every call of it
 *     clears before its decode).
 *   - Return value: MLA_OK (0) or a negative MLA_ERR_* code.  Arguments are
 *     checked on the host before anything is launched; on error nothing is
 *     launched and mla_last_error_string() (thread-local) says why.
 *   - Launches are asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).  Problems found on the device (a bounded wait
 *     that gave up, a sequence length beyond the page table) are OR-ed as
 *     MLA_STATUS_* bits into the optional device word `status`, which the
 *     caller zeroes and reads back.
 *   - Query row order is the flat [B, q_len, H] order: row r = (b*q_len+i)*H+h.
 */
#ifndef MLA_DECODE_H
#define MLA_DECODE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* mla_stream_t; /* same type as cudaStream_t */

enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = -1, /* null pointer, bad size or count */
  MLA_ERR_UNSUPPORTED = -2, /* valid but not built (e.g. page_size != 64) */
  MLA_ERR_MISALIGNED = -3,  /* a pointer breaks the stated alignment */
  MLA_ERR_CUDA = -4,        /* a CUDA runtime call or launch failed */
  MLA_ERR_PAGE_TABLE = -5,  /* mla_check_page_table found a bad entry */
  MLA_ERR_SCRATCH = -6      /* mla_decode_scratch: the call needs more than
                               the library's static scratch */
};

/* Bits OR-ed into the device status word by the kernels. */
enum {
  MLA_STATUS_WAIT_TIMEOUT = 1, /* a bounded pipeline wait gave up; outputs of
                                  that CTA are incomplete */
  MLA_STATUS_BAD_LENGTH = 2,   /* a sequence length exceeded the page table
                                  stride and was clamped */
  MLA_STATUS_BAD_SLOT = 4,     /* a page's slot run lay outside the pool; its
                                  rows were read as zeros */
  MLA_STATUS_BAD_WORK = 8      /* a work-list entry named no work unit; that
                                  cluster did nothing (see mla_plan_sched) */
};

typedef enum { MLA_KV_BF16 = 0, MLA_KV_FP8_E4M3 = 1 } mla_kv_dtype;

/* Latent row geometry ([VRAM-KV], [K3-MEM]). */
#define MLA_ROW_DIM 576   /* kv_lora_rank + qk_rope_head_dim */
#define MLA_NOPE_DIM 512  /* kv_lora_rank: c_kv, also the value */
#define MLA_ROPE_DIM 64   /* qk_rope_head_dim */
#define MLA_VALUE_DIM 512
#define MLA_QK_NOPE_DIM 128 /* per-head query/key dims before absorption */
#define MLA_V_HEAD_DIM 128  /* per-head value dims after the output projection */
#define MLA_PAGE_SIZE 64  /* the only page size the kernels are built for */
#define MLA_SCRATCH_BYTES (256u << 20) /* static scratch of mla_decode_scratch */
#define MLA_ROWS_PER_UNIT 256 /* query rows one BF16 work unit (a 4-CTA cluster) owns;
                                 an FP8 unit (a 2-CTA cluster) owns half */

/* Last error message of this thread ("" if none).  Owned by the library. */
const char* mla_last_error_string(void);

/* SM count of `device` (cudaDevAttrMultiProcessorCount), or a negative
 * MLA_ERR_* code. */
int mla_num_sms(int device);

/* Number of work units of the tensor-core decode kernel (clusters of four
 * CTAs, one CTA per SM) that can be resident at once on the current device
 * (cudaOccupancyMaxActiveClusters with the kernel's cluster size, block size
 * and shared memory), or a negative MLA_ERR_*. */
int mla_cluster_slots(void);

/*
 * The pages' split rule, reproduced for comparison ([K3-MLA]):
 *   split = max(1, min(148 // B // (q_len * 2), 32)).
 * The floor of 1 is implied by the same paragraph ("split = 1 for B >= 8").
 * Returns the split count, or MLA_ERR_INVALID_ARG for B < 1 or q_len < 1.
 */
int mla_plan_heuristic(int B, int q_len);

/*
 * Wave-rounding split planner (replaces the rule above; [K3-MLA] shows that
 * rule leaving a partial second wave).  Work units are decode clusters, one
 * per (virtual request v, split s, row unit u) with U = ceil(H*q_len /
 * rows_per_unit) row units, launched split-major (s slowest, then v, u
 * fastest): the BF16
 * kernel serves 256 rows with a 4-CTA cluster, the FP8 kernel 128 rows with
 * a 2-CTA cluster.  For every S in [1, s_max] the unit costs
 * pages(v, s) + c0 page tiles, where request v's P_v = ceil(L_v / 64) pages
 * are dealt as floor((s+1) P_v / S) - floor(s P_v / S); the units are list-
 * scheduled onto `slots` cluster slots in launch order; the objective is
 *   J(S) = makespan(S) + lam * S * rows / 1024,   rows = V * q_len * H,
 * (the second term prices the partial outputs each extra split writes and
 * the combine re-reads).  The smallest J wins, ties go to fewer splits.
 * All three planners skip a candidate whose lower bound max(total cost /
 * slots, largest unit cost) + its split price cannot beat the best J so far,
 * and stop a schedule once it reaches that J: the result is the full
 * search's (about 0.2 ms of host time for 16 requests, 2 ms for 1024
 * virtual requests, on 36 slots).
 *   rows_per_unit  query rows per work unit (> 0)
 *   seq_lens_host  host int32 [V] (V = num_shards * B virtual requests)
 *   slots          concurrent cluster slots (> 0)
 *   s_max          largest split count considered (1..1024)
 *   num_splits_out chosen S;  wave_eff_out: sum(unit cost)/(slots*makespan);
 *   makespan_out   makespan in page tiles (may be NULL)
 */
int mla_plan_ex(int V, int q_len, int H, int rows_per_unit,
                const int32_t* seq_lens_host, int slots, int s_max, double c0,
                double lam, int* num_splits_out, float* wave_eff_out,
                double* makespan_out);

/*
 * mla_plan_ex with the library's defaults for the kernel that serves
 * kv_dtype: BF16 -> rows_per_unit = 256 and slots = mla_cluster_slots() (or
 * num_sms / 4 when num_sms > 0); FP8 E4M3 -> rows_per_unit = 128 and the
 * resident 2-CTA clusters of the FP8 kernel (or num_sms / 2); s_max = 64;
 * c0 = 16 for BF16 and 32 for FP8 E4M3; lam = 1 (fitted to the kernels'
 * measured times on GB300, B = 1..24 requests x 100k / 400k tokens: a work
 * unit costs about that many pages beyond its own).
 *   B, num_shards  requests and context shards (V = B * num_shards);
 *   kv_dtype       MLA_KV_BF16 or MLA_KV_FP8_E4M3 (else MLA_ERR_INVALID_ARG)
 *   seq_lens_host  host int32 [num_shards * B] (shard-local lengths).
 */
int mla_plan(int B, int q_len, int H, int num_shards, mla_kv_dtype kv_dtype,
             const int32_t* seq_lens_host, int num_sms, int* num_splits_out,
             float* wave_eff_out);

/*
 * Split planner with per-request boundaries (work balanced over the resident
 * clusters, [K3-MLA]'s wave-aware rounding taken further).  Candidates, all
 * scored like mla_plan_ex (list scheduling of the work units on `slots` in
 * launch order, which is part-major: every request's part s before any part
 * s + 1; a unit costs its pages + c0, an empty unit 1; J = makespan +
 * lam * S * rows / 1024), the first of equal J kept:
 *   1. the uniform deal for S = 1 .. s_max;
 *   2. for S = 2 .. max_parts and 32 caps b = ceil(Pmax * k / 32): part 0 of
 *      request v = min(P_v, b) pages, the other P_v - part0 pages dealt
 *      over parts 1 .. S-1 (boundary m = part0 + floor((m-1) rest / (S-1)));
 *   3. for S = 2 .. max_parts, equal chunks of u = ceil(Pmax / S) pages:
 *      boundary m of request v = min(P_v, m u), so a ragged batch gets units
 *      of equal work (long requests more parts, short ones fewer).
 * Writes S = *num_parts_out and the boundaries as [V][S + 1] int32 at the
 * start of split_pages_out (a HOST buffer of at least V * (s_max + 1)
 * entries), for mla_decode_partial's split_pages.
 *   rows_per_unit, seq_lens_host, slots, s_max, c0, lam: as mla_plan_ex
 *   max_parts      largest part count of families 2 and 3 (1..s_max)
 *   wave_eff_out   sum(unit cost) / (slots * makespan), may be NULL
 *   makespan_out   makespan in pages, may be NULL
 */
int mla_plan_parts_ex(int V, int q_len, int H, int rows_per_unit,
                      const int32_t* seq_lens_host, int slots, int s_max,
                      int max_parts, double c0, double lam,
                      int32_t* split_pages_out, int* num_parts_out,
                      float* wave_eff_out, double* makespan_out);

/*
 * mla_plan_parts_ex with mla_plan's defaults (rows per unit and slots of the
 * kernel that serves kv_dtype, s_max = 64, c0 and lam as mla_plan).
 * split_pages_out: HOST int32 buffer of at least num_shards * B * 65 entries.
 */
int mla_plan_parts(int B, int q_len, int H, int num_shards,
                   mla_kv_dtype kv_dtype, const int32_t* seq_lens_host,
                   int num_sms, int max_parts, int32_t* split_pages_out,
                   int* num_parts_out, float* wave_eff_out);

/*
 * Work-balanced scheduler: the parts of mla_plan_parts_ex plus the order in
 * which the kernel takes its work units.  A work unit is one part s of one
 * virtual request v for one group u of rows_per_unit query rows, identified
 * by id = (s * V + v) * U + u, U = ceil(q_len * H / rows_per_unit); without
 * a work list the kernel launches the ids in increasing order.  Here the
 * units are ordered longest first (cost = pages + c0, an empty unit 1; equal
 * costs in increasing id), so the cluster slots, which the hardware fills in
 * launch order as they free up, run a longest-processing-time list schedule:
 * on a ragged batch the long parts start first and the short ones fill the
 * gaps at the end ([K3-MLA]'s wave-aware rounding, taken to unequal work).
 * Candidates are the three families of mla_plan_parts_ex, each scored by the
 * makespan of that schedule plus lam * S * rows / 1024; the first of equal
 * scores is kept.
 *   V .. lam, split_pages_out, num_parts_out: as mla_plan_parts_ex
 *   work_out       HOST int32 buffer of work_capacity entries; receives the
 *                  V * S * U unit ids in launch order (a permutation of
 *                  0 .. V*S*U - 1), for the decode entry points' `work`
 *   num_work_out   V * S * U
 *   wave_eff_out   sum(unit cost) / (slots * makespan), may be NULL
 *   makespan_out   makespan in pages, may be NULL
 * MLA_ERR_INVALID_ARG (nothing written) if work_capacity < V * S * U.
 */
int mla_plan_sched_ex(int V, int q_len, int H, int rows_per_unit,
                      const int32_t* seq_lens_host, int slots, int s_max,
                      int max_parts, double c0, double lam,
                      int32_t* split_pages_out, int* num_parts_out,
                      int32_t* work_out, int64_t work_capacity,
                      int64_t* num_work_out, float* wave_eff_out,
                      double* makespan_out);

/*
 * mla_plan_sched_ex with mla_plan's defaults (rows per unit and slots of the
 * kernel that serves kv_dtype, s_max = 64, c0 and lam as mla_plan).
 * split_pages_out: HOST int32 [num_shards * B * 65]; work_out: HOST int32
 * [work_capacity], at most num_shards * B * 64 * ceil(q_len * H / 128)
 * entries are written.
 */
int mla_plan_sched(int B, int q_len, int H, int num_shards,
                   mla_kv_dtype kv_dtype, const int32_t* seq_lens_host,
                   int num_sms, int max_parts, int32_t* split_pages_out,
                   int* num_parts_out, int32_t* work_out,
                   int64_t work_capacity, int64_t* num_work_out,
                   float* wave_eff_out);

/*
 * Host-side check of a page table (optional validation mode).  All
 * pointers are HOST copies.  Checks, for every virtual request v < V:
 * 1 <= q_len; 0 <= seq_lens[v] <= stride; without kv_limit seq_lens[v] >=
 * q_len; with kv_limit 0 <= kv_limit[v, i] <= seq_lens[v]; every entry
 * t < seq_lens[v] is a slot in [0, num_slots); every page is one contiguous,
 * page-aligned run: req_to_token[v, t] == req_to_token[v, 64*(t/64)] + t%64
 * and req_to_token[v, 64*(t/64)] % 64 == 0.  The decode kernels read only the
 * first entry of each page and rely on these properties.
 * Returns MLA_OK or MLA_ERR_PAGE_TABLE / MLA_ERR_INVALID_ARG with a message.
 */
int mla_check_page_table(const int32_t* req_to_token_host, int64_t stride,
                         const int32_t* seq_lens_host,
                         const int32_t* kv_limit_host, int V, int q_len,
                         int page_size, int64_t num_slots);

/*
 * Partial decode ([VRAM-KV], [K3-MLA], [K3-SPLIT], [K3-INTRO]): for every
 * split s, shard c, request b, query i, head h (row r = (b*q_len+i)*H+h,
 * virtual request v = c*B + b), over the tokens of split s of v's page list
 * that query i may see (t < kv_limit[v, i], or t <= seq_lens[v] - q_len + i
 * when kv_limit is NULL):
 *   x    = [q_nope_absorbed[b,i,h,:512] ; q_rope[b,i,h,:64]]
 *   k_t  = kv_pages[req_to_token[v, t], :576]  (FP8: bytes * kv_scale[slot])
 *   s_t  = sm_scale * <x, k_t>
 *   LSE_part[s,c,b,i,h] = ln sum_t exp(s_t)            (-inf if no token)
 *   O_part[s,c,b,i,h,:] = sum_t exp(s_t - LSE) k_t[:512] (0 if no token)
 * Split s of a request with P pages covers pages [s*P/S, (s+1)*P/S), or the
 * pages of split_pages when it is given.
 *
 *   q_nope_absorbed  bf16 [B, q_len, H, 512], contiguous, 16-B aligned
 *   q_rope           bf16 [B, q_len, H, 64], contiguous, 16-B aligned
 *   kv_pages         [num_slots, 576]: bf16 (1152-B rows) or E4M3 bytes
 *                    (576-B rows); 16-B aligned; num_slots >= page_size
 *   kv_scale         fp32 [num_slots] (FP8), 16-B aligned; NULL for BF16
 *   req_to_token     int32 [num_shards*B, r2t_stride]; only the entry of the
 *                    first token of each page is read (see
 *                    mla_check_page_table for the contract)
 *   seq_lens         int32 [num_shards*B], device; counts the q_len draft
 *                    tokens already in the cache
 *   kv_limit         int32 [num_shards*B, q_len] or NULL
 *   num_shards       token-interleaved context shards sharing one Q (1 = none)
 *   page_size        must be 64 (else MLA_ERR_UNSUPPORTED)
 *   sm_scale         softmax scale, finite and > 0 (1/sqrt(192) for the
 *                    192-d pre-absorption query/key head)
 *   num_splits       KV splits per request, >= 1 (see mla_plan)
 *   split_pages      device int32 [num_shards*B, num_splits + 1] or NULL:
 *                    part s of virtual request v covers pages
 *                    [split_pages[v][s], split_pages[v][s+1]) (clamped to
 *                    [0, ceil(L_v / 64)]; empty when the upper bound is not
 *                    above the lower; see mla_plan_parts).  The rows must
 *                    partition each request's pages (non-decreasing from 0
 *                    to ceil(L_v / 64)) for the combine to be the full
 *                    result; NULL deals the pages uniformly.
 *                    Without a work list, work is launched split by split
 *                    (all first parts, then all second parts, ...).
 *   work             device int32 [num_work] or NULL: the work-unit ids
 *                    (see mla_plan_sched) in launch order.  It must hold
 *                    every id 0 .. num_work - 1 once, num_work = num_splits *
 *                    num_shards * B * ceil(q_len * H / R), R = 256 rows for
 *                    BF16 KV and 128 for FP8 (else MLA_ERR_INVALID_ARG); an
 *                    entry outside that range sets MLA_STATUS_BAD_WORK and
 *                    its cluster does nothing.  The results do not depend on
 *                    the order.
 *   num_work         entries of work (0 when work is NULL)
 *   O_part           fp32 [num_splits, num_shards, B, q_len, H, 512], 16-B al.
 *   LSE_part         fp32 [num_splits, num_shards, B, q_len, H]
 *   status           device int or NULL (MLA_STATUS_* bits are OR-ed in)
 * Rows of slots beyond a request's length (the tail of its last page) are
 * never used, whatever they hold.  A token that query i may not see adds
 * nothing to its rows, whatever the token's row holds (NaN included): the
 * rows of query i are bitwise those of a cache without that token.  A NaN
 * score that a row does see makes that row NaN (O_part and LSE_part), as the
 * definition gives.
 * Precision with FP8 KV: the contractions run on FP8 tensor cores over the
 * stored E4M3 bytes.  Query elements above 32x their row's mean |q|
 * (outlier channels, up to 4 per group of 128 rows, shared by the group)
 * leave the 8-bit representation and are multiplied with the key bytes in
 * fp32, exactly.  The rest of each row is represented as 2^e (hi + lo), two
 * E4M3 parts with a power-of-two row scale: exact for every element at least
 * 2^-9 of the row's largest remaining |q|, off by at most 2^-17 of it
 * otherwise (a fifth outlier channel in one group stays in this split).  The
 * probabilities (times the token's scale) are represented as E4M3 + E5M2
 * parts, 2^-7 relative error at most.  kv_scale must be finite; its
 * magnitude may lie anywhere in [2^-100, 2^100].
 */
int mla_decode_partial(const void* q_nope_absorbed, const void* q_rope,
                       const void* kv_pages, const float* kv_scale,
                       mla_kv_dtype kv_dtype, int64_t num_slots,
                       const int32_t* req_to_token, int64_t r2t_stride,
                       const int32_t* seq_lens, const int32_t* kv_limit,
                       int B, int q_len, int H, int num_shards, int page_size,
                       float sm_scale, int num_splits,
                       const int32_t* split_pages, const int32_t* work,
                       int num_work, float* O_part, float* LSE_part,
                       int* status, mla_stream_t stream);

/*
 * mla_decode_partial with bf16 partial outputs: the same computation and
 * arguments, but O_part is bf16 [num_splits, num_shards, B, q_len, H, 512],
 * 16-B aligned, each normalised value rounded to nearest even from fp32
 * (the survey's A7 step allows a bf16 O_part; LSE_part stays fp32).  Half
 * the bytes of the epilogue's stores and of the combine's reads; each part
 * gains at most 2^-9 relative rounding before the merge.  BF16 and FP8 KV
 * (tensor-core kernels).  Merge with mla_lse_combine_bf16_parts.
 */
int mla_decode_partial_bf16_parts(
    const void* q_nope_absorbed, const void* q_rope, const void* kv_pages,
    const float* kv_scale, mla_kv_dtype kv_dtype, int64_t num_slots,
    const int32_t* req_to_token, int64_t r2t_stride, const int32_t* seq_lens,
    const int32_t* kv_limit, int B, int q_len, int H, int num_shards,
    int page_size, float sm_scale, int num_splits, const int32_t* split_pages,
    const int32_t* work, int num_work, void* O_part, float* LSE_part,
    int* status, mla_stream_t stream);

/*
 * Whole decode in one launch ([K3-MLA]: the partial (O, LSE) per split and
 * shard, then dcp_lse_combine): mla_decode_partial followed by the
 * mla_lse_combine over its num_splits * num_shards parts, fused.  Each
 * cluster counts its arrival for its (request, row unit) once its part is
 * written; the cluster that completes the count merges that unit's rows and
 * resets the count, so no cluster ever waits for another.
 *   inputs as mla_decode_partial; O_part and LSE_part are the caller's
 *                    workspace for the parts (same sizes)
 *   counters   device int32 [B * ceil(q_len * H / 128)], 4-B aligned:
 *              all zero before the call; every call leaves them zero (also
 *              when a bounded wait timed out) as long as its work list
 *              holds every unit once; after a call that set
 *              MLA_STATUS_BAD_WORK, zero them again.  Two calls that may run
 *              at the same time must not share counters or workspace.
 *   out        bf16 [B, q_len, H, 512] (round to nearest even), 16-B aligned
 *   lse_out    fp32 [B, q_len, H] (natural log) or NULL
 * Same errors as mla_decode_partial; MLA_ERR_INVALID_ARG if counters or out
 * is NULL.  The tensor-core kernels only (page_size 64).
 */
int mla_decode(const void* q_nope_absorbed, const void* q_rope,
               const void* kv_pages, const float* kv_scale,
               mla_kv_dtype kv_dtype, int64_t num_slots,
               const int32_t* req_to_token, int64_t r2t_stride,
               const int32_t* seq_lens, const int32_t* kv_limit, int B,
               int q_len, int H, int num_shards, int page_size, float sm_scale,
               int num_splits, const int32_t* split_pages,
               const int32_t* work, int num_work, float* O_part,
               float* LSE_part, int32_t* counters, void* out, float* lse_out,
               int* status, mla_stream_t stream);

/*
 * mla_decode with no workspace argument and no allocation: the arrival
 * counters and the per-part (O, LSE) results live in one static device array
 * of the library (MLA_SCRATCH_BYTES, 256-byte aligned, one per device),
 * whose address is looked up with cudaGetSymbolAddress by the first call on
 * each device (make that first call before any stream capture; the address
 * is kept for the life of the process, so do not call this again on a
 * device after cudaDeviceReset).  Each call first clears the counters on
 * its stream (cudaMemsetAsync, no allocation), so a call that left them
 * non-zero (a work list naming no unit or one unit twice, a timed-out wait)
 * does not affect the next.  The call makes no cudaMalloc or cudaFree.  The
 * pages have no counterpart: their kernels take their workspace from the
 * serving framework; this entry point is the library's own, for callers that
 * hold no workspace.
 *   arguments     as mla_decode, without O_part, LSE_part and counters
 * Size limit: the call needs mla_scratch_bytes(B, q_len, H, num_shards,
 * num_splits) bytes; above MLA_SCRATCH_BYTES it returns MLA_ERR_SCRATCH
 * (checked before every other argument, nothing launched) and
 * mla_last_error_string() gives both sizes.
 * Races: every call on a device uses the same array.  Calls that may run at
 * the same time on one device (two streams not ordered by events, two host
 * threads) race on it: the counters may then complete a unit early and the
 * merged outputs and the counters' zero state are lost.  Order such calls
 * (one stream, or events) or use mla_decode with separate workspace.
 */
int mla_decode_scratch(const void* q_nope_absorbed, const void* q_rope,
                       const void* kv_pages, const float* kv_scale,
                       mla_kv_dtype kv_dtype, int64_t num_slots,
                       const int32_t* req_to_token, int64_t r2t_stride,
                       const int32_t* seq_lens, const int32_t* kv_limit, int B,
                       int q_len, int H, int num_shards, int page_size,
                       float sm_scale, int num_splits,
                       const int32_t* split_pages, const int32_t* work,
                       int num_work, void* out, float* lse_out, int* status,
                       mla_stream_t stream);

/* Scratch bytes mla_decode_scratch needs for this shape (each of the
 * counters, LSE parts and O parts rounded up to 256 bytes), or a negative
 * MLA_ERR_INVALID_ARG for a count below 1. */
int64_t mla_scratch_bytes(int B, int q_len, int H, int num_shards,
                          int num_splits);

/*
 * Cache write ([VRAM-KV], [VRAM-POOL]): store n new tokens' latent rows in
 * the paged pool, row r at slot slots[r] (the token's req_to_token entry).
 *   rows       bf16 [n, 576] (c_kv 512 then RoPE key 64), 16-B aligned
 *   slots      int32 [n], device; a slot outside [0, num_slots) is skipped
 *              and MLA_STATUS_BAD_SLOT is OR-ed into status
 *   kv_pages   [num_slots, 576] bf16 or E4M3 bytes, 16-B aligned
 *   kv_scale   fp32 [num_slots] for FP8 (NULL for BF16)
 * BF16: the rows are copied.  FP8 E4M3 (the per-token scale format; the
 * pages fix neither the scale rule nor the rounding, the reading taken is):
 *   scale = fl32(max_d |x_d| / 448); code_d = E4M3(fl32(x_d / scale)), both
 *   IEEE round-to-nearest divisions, E4M3 rounded to nearest even and
 *   saturated to +-448; an all-zero row gets scale 0 and codes 0.
 * Rows must be finite.  n = 0 is a no-op.  Slots written by two rows of one
 * call get either row.
 */
int mla_kv_write(const void* rows, int64_t n, const int32_t* slots,
                 void* kv_pages, mla_kv_dtype kv_dtype, float* kv_scale,
                 int64_t num_slots, int* status, mla_stream_t stream);

/*
 * The per-head projections around the absorbed decode ([K3-MEM]: w_kc is
 * 96 x 128 x 512 bf16 and the absorbed query 512-d; the pages' kv_b_proj is
 * absorbed into w_kc and w_vc, mla_prepare is the step before the decode).
 * Rows m = b * q_len + i, M = B * q_len; fp32 accumulation, bf16 results
 * rounded to nearest even.
 *   mla_absorb_q:    q_absorbed[m, h, :512] = q_nope[m, h, :128] . w_kc[h]
 *     q_nope bf16 [M, H, 128]; w_kc bf16 [H, 128, 512]; q_absorbed bf16
 *     [M, H, 512] (the q_nope_absorbed input of the decode)
 *   mla_project_out: o_v[m, h, :128] = o_latent[m, h, :512] . w_vc[h]
 *     o_latent bf16 [M, H, 512] (the decode's out); w_vc bf16 [H, 512, 128]
 *     (reading: v_head_dim 128, the pages give w_vc's name only); o_v bf16
 *     [M, H, 128]
 * All arrays device, contiguous, 16-B aligned; H >= 1, M >= 1, and
 * ceil(M / 128) * H * 4 < 2^31 (else MLA_ERR_INVALID_ARG).  Launched with
 * programmatic dependent launch: the kernel starts while the stream's
 * previous kernels finish, prefetches its weights into L2, and waits for
 * them before it reads any input or writes any output.
 * A bounded wait that gives up sets MLA_STATUS_WAIT_TIMEOUT in status.
 */
int mla_absorb_q(const void* q_nope, const void* w_kc, void* q_absorbed, int M,
                 int H, int* status, mla_stream_t stream);
int mla_project_out(const void* o_latent, const void* w_vc, void* o_v, int M,
                    int H, int* status, mla_stream_t stream);

/*
 * The same computation on plain CUDA cores (no tensor cores, no TMA): a
 * slow, simple GPU kernel kept to cross-check the tensor-core path and to
 * cover shapes it does not take.  Same arguments and outputs.
 */
int mla_decode_partial_simt(const void* q_nope_absorbed, const void* q_rope,
                            const void* kv_pages, const float* kv_scale,
                            mla_kv_dtype kv_dtype, int64_t num_slots,
                            const int32_t* req_to_token, int64_t r2t_stride,
                            const int32_t* seq_lens, const int32_t* kv_limit,
                            int B, int q_len, int H, int num_shards,
                            int page_size, float sm_scale, int num_splits,
                            const int32_t* split_pages,
                            float* O_part, float* LSE_part, int* status,
                            mla_stream_t stream);

/*
 * LSE combine ([K3-MLA], dcp_lse_combine): for each of `rows` rows, over the
 * num_parts partials (part j at O_part + j*rows*512, LSE_part + j*rows):
 *   M = max_j LSE_j; w_j = exp(LSE_j - M) (parts with LSE = -inf skipped);
 *   out = sum_j w_j O_j / sum_j w_j;  lse_out = M + ln sum_j w_j.
 * All parts empty: out = 0, lse_out = -inf.  A part with LSE = NaN makes the
 * row NaN (out and lse_out).
 *   O_part   fp32 [num_parts, rows, 512], 16-B aligned
 *   LSE_part fp32 [num_parts, rows]
 *   out      bf16 [rows, 512] (round to nearest even), 16-B aligned
 *   lse_out  fp32 [rows] or NULL
 * With mla_decode_partial's layout, num_parts = num_splits * num_shards and
 * rows = B * q_len * H.
 */
int mla_lse_combine(const float* O_part, const float* LSE_part, int num_parts,
                    int64_t rows, void* out, float* lse_out,
                    mla_stream_t stream);

/*
 * The same merge over bf16 parts (O_part bf16 [num_parts, rows, 512], 16-B
 * aligned, as mla_decode_partial_bf16_parts writes them), each value widened
 * exactly to fp32 before the weighted sum.
 */
int mla_lse_combine_bf16_parts(const void* O_part, const float* LSE_part,
                               int num_parts, int64_t rows, void* out,
                               float* lse_out, mla_stream_t stream);

/*
 * Page-table gather through the decode kernel's own TMA path (for the
 * bit-exact test of the gather): copies the raw bytes of token t's row,
 * kv_pages[req_to_token[v, t]], for t < seq_lens[v], into
 * dense_out[row_offset[v] + t, :].
 *   row_offset  int64 [V] device, the first dense row of each request
 *   dense_out   [sum_v seq_lens[v], 576] of the KV element type, 16-B al.
 */
int mla_debug_gather(const void* kv_pages, mla_kv_dtype kv_dtype,
                     int64_t num_slots, const int32_t* req_to_token,
                     int64_t r2t_stride, const int32_t* seq_lens,
                     const int64_t* row_offset, int V, int page_size,
                     void* dense_out, mla_stream_t stream);

/*
 * Test entry point of the bounded waits (the pages define no failure
 * handling; this is the library's own).  Every pipeline wait of the decode
 * kernels gives up after 2 s of %globaltimer, or as soon as another warp of
 * its CTA has given up (the CTA's abort flag), and then sets
 * MLA_STATUS_WAIT_TIMEOUT instead of spinning on.  This launches one CTA of
 * 64 threads whose thread 0 runs that same wait on a barrier phase that
 *   mode 0: nothing completes: the wait gives up after its 2 s limit and
 *           MLA_STATUS_WAIT_TIMEOUT is OR-ed into *status;
 *   mode 1: nothing completes, but another warp raises the CTA's abort flag
 *           after delay_us: the wait gives up then, status as in mode 0;
 *   mode 2: another warp completes after delay_us: the wait succeeds and
 *           *status is not touched.
 *   delay_us    in [0, 1000000] (else MLA_ERR_INVALID_ARG)
 *   status      device int, 4-B aligned (required)
 *   elapsed_ns  device uint64, 8-B aligned (required): the wait's duration
 * The kernel holds no tensor memory and starts no TMA, bulk copy or MMA, so
 * it always ends and leaves the context usable.
 */
int mla_debug_wait(int mode, int delay_us, int* status, uint64_t* elapsed_ns,
                   mla_stream_t stream);

/*
 * Test entry point of the FP8 cache write's division (mla_kv_write): the
 * write forms each code's quotient x / scale from one correctly rounded
 * reciprocal of the row's scale and one Markstein correction instead of an
 * IEEE division per element.  This runs that routine against the IEEE
 * division for every positive finite bf16 row maximum amax (scale =
 * fl32(amax / 448); scales outside [2^-90, 2^120], where the write divides
 * directly, are skipped) and every bf16 element x with |x| <= amax, and adds to
 * the two device counters (uint64, zeroed by the caller) the cases where
 * quotients of magnitude 2^-11 or more differ in any bit, and where the
 * E4M3 codes differ.  Both stay 0 for a correct build.  No counterpart on
 * the pages (a property of the quantiser the reading of the pages fixes).
 * Errors: NULL counter -> MLA_ERR_INVALID_ARG; misaligned -> MLA_ERR_MISALIGNED.
 */
int mla_debug_quotients(uint64_t* bit_mismatches, uint64_t* code_mismatches,
                        mla_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MLA_DECODE_H */
