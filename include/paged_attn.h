/*
 * paged_attn.h — C ABI of the GB300 (sm_103a) paged-attention library.
 *
 * The operation: for every query token i of sequence b and every query head h,
 * attend over that sequence's keys, which live in a pool of fixed-size pages
 * reached through a per-sequence block table.  Scores are scale * q.k; key j is
 * valid iff j < seq_lens[b] and, when causal, j <= q_offset[b] + i; the softmax
 * of the valid scores weights the V rows.  The keys may be split into split_kv
 * partitions, each giving a normalised partial output plus its log-sum-exp,
 * which paged_attn_combine merges.
 *
 * Sources (page titles and sections):
 *   rocm-libraries PR #14349 (gfx942 tiled-2D attention), Motivation and
 *     Technical Details: paged K/V through a block table; pages of page_size
 *     tokens holding every kv head; 64-bit page bases for pools past 2^31
 *     bytes; page ids loaded once per tile; GQA head groups.
 *   rocMLIR PR #2220 "Paged Attention: migraphx & highlevel pipeline changes":
 *     attention whose K/V arrive through an address view of paged storage.
 *   rocMLIR PR #2371 "Fix split-kv attention masking...", Technical Details:
 *     ceil-divided split partition with clamped (empty) trailing splits; the
 *     -inf - (-inf) guard; the 0/0 guard; per-row causal reach with the prefix
 *     offset; an f32 combine for narrow float types.
 *
 * Conventions shared by every call
 *   - All tensor pointers are DEVICE pointers, row-major and 16-byte aligned;
 *     every tensor is dense except q, whose tokens may be further apart
 *     (pa_dims.q_stride).  The caller owns every buffer; the library
 *     allocates nothing.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  The returned status reports argument validation and launch
 *     errors only; faults inside a kernel surface on the stream as CUDA errors.
 *   - Block-table slots at or past ceil(seq_lens[b] / page_size) are never
 *     read, so they may hold anything (-1, 0x7FFFFFFF, garbage).
 *   - A page id that is read and lies outside [0, num_pages) is not
 *     dereferenced: its tokens read as zero and bit PA_ERRBIT_PAGE_RANGE is set
 *     in the device error word (see paged_attn_last_error_word).
 */
#ifndef PAGED_ATTN_H
#define PAGED_ATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element types (PA_FP8_E4M3, PA_INT8: quantized K/V pools only, see paged_attn_fwd_kvq) */
enum { PA_F32 = 0, PA_F16 = 1, PA_BF16 = 2, PA_FP8_E4M3 = 3, PA_INT8 = 4 };

/* status codes */
enum {
    PA_OK = 0,
    PA_EINVAL = -1,        /* inconsistent or out-of-range argument */
    PA_EDTYPE = -2,        /* unsupported element type */
    PA_EUNSUPPORTED = -3,  /* shape outside the supported envelope (or forced variant cannot run it) */
    PA_ECUDA = -4,         /* a CUDA runtime/driver call failed */
    PA_EBOUNDS = -5,       /* paged_attn_last_error_word: a page id outside [0, num_pages) was read */
    PA_ETIMEOUT = -6       /* paged_attn_last_error_word: a pipeline wait gave up; outputs are invalid */
};

/* bits of the device error word */
enum {
    PA_ERRBIT_PAGE_RANGE = 1u,   /* a block-table page id used by a sequence was outside [0, num_pages) */
    PA_ERRBIT_TIMEOUT = 2u,      /* a pipeline wait gave up after its time limit (results invalid) */
    PA_ERRBIT_SEQ_CLIPPED = 4u,  /* seq_lens[b] needed more pages than bt_stride holds; clipped to bt_stride pages */
    PA_ERRBIT_QSTART = 8u        /* paged_attn_fwd_varlen: a q_start entry out of [0, total tokens] or decreasing */
};

/* kernel variants (paged_attn_fwd_variant) */
enum {
    PA_VARIANT_AUTO = 0,         /* planner's choice */
    PA_VARIANT_SIMT = 1,         /* CUDA cores: any dtype, any head grouping (a single query row per kv head
                                    in bf16/f16 at head_dim 64/128 streams K/V through a TMA ring) */
    PA_VARIANT_MMA_DECODE = 2,   /* tensor-core decode: Sq * (Hq/Hkv) <= 16 rows, keys split across warps */
    PA_VARIANT_MMA_PREFILL = 3,  /* warp-level tensor cores, 64-row query tiles (prefill / long query runs) */
    PA_VARIANT_TC05_PREFILL = 4, /* tcgen05 + tensor memory, 128-row query tiles; bf16/f16, head_dim 128,
                                    Hq/Hkv dividing 128, scale > 0 (the planner sends scale <= 0 to
                                    PA_VARIANT_MMA_PREFILL) */
    PA_VARIANT_MMA_T = 5,        /* tensor cores, transposed products (keys and head dim as MMA rows), 8-row
                                    units; bf16/f16, head_dim 256 (the only 16-bit variant there) */
    PA_VARIANT_MMA_SPLIT_GROUP = 6 /* tensor-core decode (Sq * (Hq/Hkv) <= 16 rows, head_dim 64/128, bf16/f16)
                                    with short splits: a CTA per four consecutive splits, one warp per split;
                                    every split at most 8 pages (ceil(bt_stride / split_kv) <= 8).  The
                                    planner takes it when that holds and one CTA per split would need more
                                    than two CTAs per multiprocessor */
};

/*
 * Problem shape.
 *   q            [batch, q_len, num_q_heads, head_dim]               (dtype)
 *   k/v pools    [num_pages, page_size, num_kv_heads, head_dim]      (dtype)
 *   block_table  [batch, bt_stride] int32; row b lists the physical pages of
 *                sequence b in logical order
 *   seq_lens     [batch] int32: valid K/V tokens of sequence b, including its
 *                q_len newest tokens
 *   q_offset     [batch] int32 or NULL: position of query row 0 of sequence b
 *                inside its K/V sequence (NULL means seq_lens[b] - q_len)
 * Layouts: the heads of one query token are dense (head h at h * head_dim); consecutive tokens are
 * q_stride elements apart (q_stride = 0: dense, num_q_heads * head_dim), and sequence b's token i is
 * token b * q_len + i (a variable-length batch's packed token t is token t).  Every other tensor
 * (out, lse, partials, pools, block table rows within bt_stride) is dense.
 * Supported: dtype in {PA_F32, PA_F16, PA_BF16}; head_dim in {64, 128, 256} (256: not for the FP8 and
 * variable-length entry points);
 * page_size in {16, 32, 64}; num_q_heads a multiple of num_kv_heads;
 * num_pages * page_size < 2^31 tokens (each pool may exceed 2^31 bytes).
 */
typedef struct pa_dims {
    int32_t batch;         /* B */
    int32_t q_len;         /* Sq */
    int32_t num_q_heads;   /* Hq */
    int32_t num_kv_heads;  /* Hkv */
    int32_t head_dim;      /* D */
    int32_t page_size;     /* tokens per page */
    int64_t num_pages;     /* pages in each of the K and V pools */
    int32_t bt_stride;     /* elements between consecutive block-table rows */
    int32_t dtype;         /* PA_F32 / PA_F16 / PA_BF16 */
    int64_t q_stride;      /* elements between consecutive query tokens of q; 0 = dense
                              (num_q_heads * head_dim).  A larger stride reads q as a view, for
                              example of a fused QKV projection's output; a multiple of
                              16 bytes / element size (8 for 16-bit q, 4 for f32) */
} pa_dims;

/*
 * paged_attn_fwd — attention over the paged K/V cache, per split partition.
 *
 * split_kv = S >= 1.  Sequence b's nblk = ceil(seq_lens[b] / page_size) pages
 * are cut into S runs of per = ceil(nblk / S) pages; run s covers pages
 * [min(s*per, nblk), min((s+1)*per, nblk)), so trailing runs may be empty
 * (rocMLIR PR #2371, split-KV iteration math).
 *
 * scale multiplies q.k.  Outputs:
 *   S == 1: out [B, Sq, Hq, D] in dtype (round to nearest even);
 *           lse [B, Sq, Hq] float32 natural-log sum-exp, or NULL.
 *   S >  1: out [S, B, Sq, Hq, D] float32 per-split outputs, each normalised by
 *           its own softmax sum; lse [S, B, Sq, Hq] float32 (required).
 * A row with no valid key in a partition gets lse -inf, never NaN, and output 0
 * (rocMLIR PR #2371, the -inf - (-inf) and 0/0 guards).  With S > 1 such a row's
 * partial output is not always written (the prefill kernel skips the rows of a tile
 * that its split's keys do not reach): read a partial row only where its lse is
 * finite, as paged_attn_combine does (it gives weight 0 to a row with lse -inf).
 * Returns PA_OK or a negative status; nothing is launched on error.
 */
int paged_attn_fwd(const void *q, const void *k_cache, const void *v_cache, const int32_t *block_table,
                   const int32_t *seq_lens, int causal, const int32_t *q_offset, int split_kv, float scale,
                   void *out, float *lse, const pa_dims *dims, void *stream);

/* paged_attn_fwd with a forced kernel variant (PA_VARIANT_*); PA_EUNSUPPORTED
 * if that variant cannot run the shape or dtype.  Same arguments otherwise. */
int paged_attn_fwd_variant(const void *q, const void *k_cache, const void *v_cache, const int32_t *block_table,
                           const int32_t *seq_lens, int causal, const int32_t *q_offset, int split_kv,
                           float scale, void *out, float *lse, const pa_dims *dims, int variant, void *stream);

/*
 * paged_attn_combine — merge split partials (rocMLIR PR #2371, f32 combine).
 *   part_out [S, rows, head_dim] float32, part_lse [S, rows] float32, where
 *   rows = B * Sq * Hq.  For each row: M = max_s lse_s; w_s = exp(lse_s - M);
 *   out = sum_s w_s O_s / sum_s w_s in float32, stored in out_dtype (round to
 *   nearest even); lse = M + log(sum_s w_s).  M = -inf gives out 0, lse -inf.
 *   out [rows, head_dim] (out_dtype); lse [rows] float32 or NULL.
 */
int paged_attn_combine(const float *part_out, const float *part_lse, int split_kv, int64_t rows, int head_dim,
                       int out_dtype, void *out, float *lse, void *stream);

/*
 * Workspace and automatic split (rocMLIR PR #2371, "device-memory-aware split-KV prefilter": the
 * extra split-KV storage is bounded by a budget of device memory / 8, clamped to [1 GiB, 8 GiB]).
 *
 * paged_attn_auto_split — the split count paged_attn_fwd_splitkv uses for split_kv = 0: the smallest
 *   S that gives at least two waves of work units over `num_sms` multiprocessors (units =
 *   B * Hkv * S, times query-row tiles for long query runs), capped by bt_stride (no sequence
 *   has more pages), by 256, and by the workspace budget for `device_bytes` of device memory.
 *   Returns S >= 1, or a negative status for invalid dims.
 * paged_attn_workspace_bytes — device bytes paged_attn_fwd_splitkv needs for split_kv partitions
 *   (0 = the automatic choice for num_sms / device_bytes): 0 when S == 1, otherwise
 *   S * B * Sq * Hq * (D + 1) * 4 rounded up to 256-byte blocks.  Negative status on error.
 */
int paged_attn_auto_split(const pa_dims *dims, int num_sms, int64_t device_bytes);
int64_t paged_attn_workspace_bytes(const pa_dims *dims, int split_kv, int num_sms, int64_t device_bytes);

/*
 * paged_attn_fwd_splitkv — the whole path in one call: the split forward into `workspace` (fp32
 * partial outputs and lse), then the fp32 combine into out [B, Sq, Hq, D] (dtype) and lse
 * [B, Sq, Hq] (float32, or NULL).  split_kv = 0 picks paged_attn_auto_split(dims, num_sms,
 * device_bytes); S == 1 writes out directly and touches no workspace.  `workspace` (device, 256-byte
 * aligned, caller-owned) must hold paged_attn_workspace_bytes(...) bytes, else PA_EINVAL; its
 * contents afterwards are unspecified.  Other arguments as paged_attn_fwd.
 */
int paged_attn_fwd_splitkv(const void *q, const void *k_cache, const void *v_cache, const int32_t *block_table,
                           const int32_t *seq_lens, int causal, const int32_t *q_offset, int split_kv, float scale,
                           void *out, float *lse, const pa_dims *dims, void *workspace, int64_t workspace_bytes,
                           int num_sms, int64_t device_bytes, void *stream);

/*
 * paged_attn_fwd_splitkv_noalloc — paged_attn_fwd_splitkv for callers that cannot allocate device
 * memory at call time (a plugin whose host framework owns every device byte, or a serving loop that
 * must never reach cudaMalloc, which can synchronise the device).  The pages have no counterpart:
 * this is a deployment convenience of this library, not part of the method.
 *
 * Same arguments and results as paged_attn_fwd_splitkv minus the workspace: the split partials go
 * to a fixed array of PA_NOALLOC_SCRATCH_BYTES inside the library's device image.  A device holds
 * that array from the moment the CUDA runtime loads its module there until the process exits: under
 * lazy module loading (CUDA's default) that is this entry point's first call on the device, under
 * CUDA_MODULE_LOADING=EAGER it is when the library is first used on the device.  An explicit
 * split_kv whose partials need more than the array (paged_attn_workspace_bytes >
 * PA_NOALLOC_SCRATCH_BYTES) returns PA_EINVAL and launches nothing; pass a smaller split_kv.
 * split_kv = 0 takes paged_attn_auto_split's choice, lowered to the largest split whose partials
 * fit the array.  No call allocates device memory.
 *   - The first call on each device looks up the array's device address (cudaGetSymbolAddress);
 *     make that first call before any stream capture on that device.
 *   - The address is kept per device ordinal for the life of the process.  It belongs to the
 *     device's primary context (the one the CUDA runtime uses): calls made from another driver
 *     context on the device, or after cudaDeviceReset, would use an address that context does not
 *     map.  Use this entry point only from the primary context and never after a device reset.
 *   - All calls share the one array.  Calls that may overlap on the GPU (different streams, or
 *     different host threads) race on it: serialise them.  Nothing in it needs clearing between
 *     calls, because each call writes every partial it later reads.
 */
#define PA_NOALLOC_SCRATCH_BYTES (64ll * 1024 * 1024)
int paged_attn_fwd_splitkv_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                   const int32_t *block_table, const int32_t *seq_lens, int causal,
                                   const int32_t *q_offset, int split_kv, float scale, void *out, float *lse,
                                   const pa_dims *dims, int num_sms, int64_t device_bytes, void *stream);

/*
 * paged_attn_fwd_varlen — one call over a batch whose sequences have different numbers of query
 * tokens: decode sequences (one new token) next to prefill chunks.  The pages' rocKE entry point
 * serves such batches ("run_unified_attention_torch", rocm-libraries PR #14349, Performance); the
 * layout below is this library's.
 *   q        [T, Hq, D] (dtype): every sequence's query tokens packed; sequence b's are rows
 *            [q_start[b], q_start[b + 1]).  T = dims->q_len (the total, not a per-sequence count).
 *   q_start  [B + 1] int32, device: q_start[0] = 0, nondecreasing, q_start[B] = T.  A sequence with
 *            no query token (q_start[b] == q_start[b + 1]) is skipped.
 *   seq_lens[b] counts sequence b's K/V tokens including its query tokens; q_offset[b] places its
 *            first query token (NULL: seq_lens[b] - its query count).
 *   out      S == 1: [T, Hq, D] (dtype); S > 1: float32 [S, T, Hq, D] partials, merged by
 *            paged_attn_combine with rows = T * Hq.  lse [T, Hq] or [S, T, Hq] (as paged_attn_fwd).
 * dims->dtype is PA_BF16 or PA_F16 (PA_F32: PA_EDTYPE); every other rule is paged_attn_fwd's.
 * Sequences of at most 16 query rows (tokens x Hq/Hkv) run as decode units and longer ones as
 * 64-row tiles of the same grid; at head_dim 128 with Hq/Hkv dividing 128, scale > 0 and at most
 * 1024 sequences, those of 64 query rows or more run instead in 128-row tcgen05 tiles, a second
 * launch on the same stream (both kernels find their sequences from q_start on the device, so
 * the host never reads it).  If q_start[b] or q_start[b + 1] lies outside [0, T], or
 * q_start[b + 1] < q_start[b], sequence b is skipped (its rows are not written) and
 * PA_ERRBIT_QSTART is set; other malformed arrays give unspecified values but no access outside
 * the buffers.
 */
int paged_attn_fwd_varlen(const void *q, const void *k_cache, const void *v_cache, const int32_t *block_table,
                          const int32_t *seq_lens, const int32_t *q_start, int causal, const int32_t *q_offset,
                          int split_kv, float scale, void *out, float *lse, const pa_dims *dims, void *stream);

/*
 * Work of a variable-length batch split the way paged_attn_fwd_varlen splits it, as the caller's
 * host-side scheduler knows it (the library itself never reads q_start on the host).  This hint and
 * the calls that take it are this library's own; the pages have no counterpart.
 *   long_pairs       over the sequences of at least 64 query rows (query tokens x Hq/Hkv >= 64):
 *                    the sum over their query tokens of the keys each token attends to
 *   short_kv_tokens  over the other sequences with at least one query token: the sum of seq_lens
 * The values only steer how many SMs each kernel gets; any values give the same results.
 */
typedef struct {
    int64_t long_pairs;
    int64_t short_kv_tokens;
} pa_varlen_hint;

/*
 * paged_attn_varlen_hint — fills *hint from HOST copies of a batch's q_start [B + 1], seq_lens [B]
 * and q_offset [B] (NULL as in paged_attn_fwd_varlen), with the reach rules of paged_attn_fwd (a
 * token sees keys [0, min(seq_len, q_offset + i + 1)) when causal, all seq_len keys otherwise).
 * dims as for paged_attn_fwd_varlen (q_len = T).  Malformed q_start entries count as no tokens.
 * Returns PA_OK, or PA_EINVAL for a NULL pointer or bad dims.
 */
int paged_attn_varlen_hint(const int32_t *q_start, const int32_t *seq_lens, const int32_t *q_offset, int causal,
                           const pa_dims *dims, pa_varlen_hint *hint);

/*
 * paged_attn_fwd_varlen_overlap — paged_attn_fwd_varlen with its two kernels run at the same time
 * on disjoint SMs.  The pages' unified entry point (rocm-libraries PR #14349, Performance) serves a
 * mixed batch in one call; this one keeps the single call and runs its two kernels at once.  The tcgen05 kernel takes the sequences of at least 64 query rows and is
 * compute-bound; the other kernel is bandwidth-bound and runs on the remaining SMs.  The tcgen05
 * kernel's SM count balances its estimated time (from hint->long_pairs) against the short
 * sequences' K/V read time (from hint->short_kv_tokens), raised by 1.3 and kept within
 * [8, 3/4 of the SMs].
 * The tcgen05 kernel runs on a high-priority stream that the library creates once per device; it
 * waits for `stream`'s earlier work and `stream` waits for it, so the call keeps stream order.
 *   - The first overlapped call on a device creates that stream, which cannot happen inside a
 *     stream capture: make the first call outside any capture.  Later calls may be captured.
 *   - Every overlapped call on a device shares the one stream.  Calls from different host threads,
 *     or captures into different graphs at the same time, would interleave their work on it:
 *     serialise them.
 * Arguments and results are those of paged_attn_fwd_varlen,
 * bit for bit.  A NULL hint, a batch without sequences of both kinds, or a shape that does not
 * take the tcgen05 kernel falls back to paged_attn_fwd_varlen's two launches on `stream`.
 */
/*
 * paged_attn_varlen_overlap_share — the number of SMs paged_attn_fwd_varlen_overlap gives the
 * tcgen05 kernel for this hint on a GPU of num_sms SMs: 0 when the two kernels would run one
 * after the other (NULL hint, no work of one kind, fewer than 16 SMs), else within
 * [8, 3/4 of num_sms].  Host-only; it does not check whether the shape takes the tcgen05 kernel.
 * Bad dims or num_sms < 1: PA_EINVAL (or the dims error).
 */
int paged_attn_varlen_overlap_share(const pa_dims *dims, const pa_varlen_hint *hint, int num_sms);

int paged_attn_fwd_varlen_overlap(const void *q, const void *k_cache, const void *v_cache,
                                  const int32_t *block_table, const int32_t *seq_lens, const int32_t *q_start,
                                  int causal, const int32_t *q_offset, int split_kv, float scale, void *out,
                                  float *lse, const pa_dims *dims, const pa_varlen_hint *hint, void *stream);

/*
 * paged_attn_fwd_kvq — paged_attn_fwd over quantized K/V pools.  The pages' sweeps include i8
 * attention (rocMLIR PR #2371, Motivation; rocMLIR PR #2222, reviewed files); this library reads a
 * quantized pool as 8-bit elements with one float32 scale per (page, kv head):
 *   value of K element (page, t, kvh, e) = elem(k_cache[page, t, kvh, e]) * k_scale[page, kvh]
 * and the same for V with v_scale, where elem() decodes a byte as
 *   PA_FP8_E4M3  an FP8 E4M3 number (OCP "fn" encoding: bias 7, no infinities, S.1111.111 is NaN)
 *   PA_INT8      a two's-complement integer in [-128, 127]
 *   k_cache, v_cache  [num_pages, page_size, num_kv_heads, head_dim] bytes, 16-byte aligned
 *   k_scale, v_scale  [num_pages, num_kv_heads] float32, 4-byte aligned
 *   kv_dtype          PA_FP8_E4M3 or PA_INT8, both pools (anything else: PA_EDTYPE)
 * q, out and dims->dtype are PA_BF16 or PA_F16 (PA_F32: PA_EDTYPE).  Every other argument, the
 * split semantics and the outputs are those of paged_attn_fwd.  A page id outside [0, num_pages)
 * reads as zeros with scale 0 and sets PA_ERRBIT_PAGE_RANGE.  The scaled score is
 * scale * k_scale * q.k_stored and the weight of a V row p * v_scale, each a float32 product;
 * the stored elements enter the tensor cores unchanged.
 */
int paged_attn_fwd_kvq(const void *q, const void *k_cache, const void *v_cache, const float *k_scale,
                       const float *v_scale, int kv_dtype, const int32_t *block_table, const int32_t *seq_lens,
                       int causal, const int32_t *q_offset, int split_kv, float scale, void *out, float *lse,
                       const pa_dims *dims, void *stream);

/* paged_attn_fwd_splitkv over quantized pools: paged_attn_fwd_kvq into `workspace`, then
 * paged_attn_combine; workspace rules and split_kv = 0 as paged_attn_fwd_splitkv. */
int paged_attn_fwd_kvq_splitkv(const void *q, const void *k_cache, const void *v_cache, const float *k_scale,
                               const float *v_scale, int kv_dtype, const int32_t *block_table,
                               const int32_t *seq_lens, int causal, const int32_t *q_offset, int split_kv,
                               float scale, void *out, float *lse, const pa_dims *dims, void *workspace,
                               int64_t workspace_bytes, int num_sms, int64_t device_bytes, void *stream);

/*
 * paged_attn_plan — the split plan as data: plan [batch, split_kv, 2] int32 =
 * {first page, one past the last page} of each run (see paged_attn_fwd).
 * seq_lens is a device pointer [batch]; negative lengths count as 0.
 */
int paged_attn_plan(const int32_t *seq_lens, int batch, int page_size, int split_kv, int32_t *plan,
                    void *stream);

/*
 * paged_attn_debug_gather — logically ordered copy of one pool:
 * out [batch, out_tokens, num_kv_heads, head_dim] (dtype); token j of sequence
 * b is copied bit for bit from its page for j < min(seq_lens[b], out_tokens)
 * and written as zero bits beyond seq_lens[b] (rocMLIR PR #2222, Key Changes
 * 1: the [numPages, pageSize] -> [seqK] view).
 */
int paged_attn_debug_gather(const void *cache, const int32_t *block_table, const int32_t *seq_lens,
                            const pa_dims *dims, int out_tokens, void *out, void *stream);

/*
 * paged_attn_debug_wait_timeout — check of the kernels' failure path: one warp waits, with the same
 * bounded pipeline wait the kernels use, on a barrier that nothing completes.  After limit_us
 * microseconds (1 .. 2 000 000; PA_EINVAL otherwise) the wait gives up, sets PA_ERRBIT_TIMEOUT in the
 * device error word and the kernel returns, leaving the context usable: the way a stalled pipeline
 * ends instead of hanging the GPU.  Asynchronous on `stream`.
 */
int paged_attn_debug_wait_timeout(uint32_t limit_us, void *stream);

/*
 * paged_attn_last_error_word — synchronise the current device, then read and
 * clear its error word (PA_ERRBIT_* bits accumulated by every call since the
 * last read) into *flags.  The status says what the bits mean for the results:
 *   PA_ETIMEOUT  PA_ERRBIT_TIMEOUT is set: a pipeline wait gave up after its
 *                2 s limit and its warp left the pipeline, so outputs written
 *                since the last read are invalid (not merely inaccurate);
 *   PA_EBOUNDS   otherwise, PA_ERRBIT_PAGE_RANGE is set: a sequence's page id
 *                lay outside [0, num_pages); its tokens read as zero (the
 *                rocm-libraries PR #14349 kernel leaves this unchecked, "Not in
 *                this PR"), every other sequence's results are exact;
 *   PA_EINVAL    otherwise, PA_ERRBIT_QSTART is set (paged_attn_fwd_varlen);
 *   PA_OK        no bit other than PA_ERRBIT_SEQ_CLIPPED is set.
 * *flags holds the bits in every case but PA_ECUDA (the read failed) and
 * PA_EINVAL for a NULL flags.  The forward calls are asynchronous and cannot
 * return these themselves: a caller that must not consume invalid outputs
 * checks this status before reading them.
 */
int paged_attn_last_error_word(uint32_t *flags);

/* Human-readable text for a status code (static storage). */
const char *paged_attn_strerror(int code);

/* Text of the CUDA error behind the calling thread's most recent PA_ECUDA ("no error" if none). */
const char *paged_attn_cuda_error_string(void);

/* Library version as an integer, major * 10000 + minor * 100 + patch. */
int paged_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_ATTN_H */
