/*
 * ta.h -- C ABI of the split-KV exact attention library for B300 (sm_103a).
 *
 * The library computes exact scaled-dot-product softmax attention for
 * long-context inference on one GPU:
 *
 *   - decode: one query per (sequence, query head) against a long KV cache,
 *     computed split-KV: each KV chunk yields a partial (running max m,
 *     sum of exponentials l, unnormalised output o) and the partials are
 *     merged by a log-sum-exp tree reduction;
 *   - the merge itself, exposed for caller-supplied partials;
 *   - causal prefill: fused QK^T * scale -> softmax -> V on the tensor cores.
 *
 * Definition (Attention glossary, jisaku.com/glossary/attention, section
 * "basic concepts and operating principle"): the query's inner product with
 * each key gives a score; softmax turns scores into weights; the output is
 * the weighted mean of the value vectors.  With s_j = scale * <q, k_j> over
 * the attended keys:
 *
 *   lse = ln sum_j exp(s_j)         (natural log, in scaled-logit units)
 *   out = sum_j exp(s_j - lse) v_j
 *
 * The split into chunks and the merge are exact reformulations, not
 * approximations (Tree Attention explainer, aibr.jp/archives/143699,
 * sections 1-3: attention's log-sum-exp "energy" is reduced along the
 * sequence axis as an associative tree; section 2: the method is exact).
 *
 * Conventions for every entry point
 *   - All tensors are row-major and contiguous, in device memory unless
 *     stated, owned by the caller.  The library never frees caller memory.
 *   - Grouped-query attention: with G = Hq / Hkv, query head h reads KV
 *     head floor(h / G).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously; no entry point
 *     synchronises the device on the compute path.
 *   - Errors: every entry point returns a ta_status and never aborts the
 *     process.  Arguments are validated before anything is launched; a
 *     rejected call launches nothing.  A launch failure is reported as
 *     TA_ERR_CUDA.  ta_last_error() gives a message for the calling thread's
 *     last non-OK status.
 */
#ifndef TA_H
#define TA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TA_OK = 0,
    TA_ERR_INVALID_ARG = 1,  /* bad sizes, null or misaligned pointers   */
    TA_ERR_UNSUPPORTED = 2,  /* valid, but a shape this build has no kernel for */
    TA_ERR_WORKSPACE = 3,    /* caller workspace missing or too small     */
    TA_ERR_CUDA = 4          /* a CUDA runtime call or launch failed      */
} ta_status;

typedef enum { TA_F32 = 0, TA_BF16 = 1 } ta_dtype;

/* Device-side conditions recorded in the workspace status word (bit set). */
enum {
    TA_DEVERR_SEQLEN = 1,   /* some seqlens[b] < 0 or > S; clamped to [0, S]     */
    TA_DEVERR_TIMEOUT = 2,  /* a pipeline wait exceeded its time limit; output invalid; the
                               launch stopped, let its copies and tensor-core operations
                               finish and returned.  Clear the workspace's control region
                               (its first 16 KiB, or all of a smaller workspace) before it is
                               used again; ta_decode_status does this for the library's own
                               workspace. */
    TA_DEVERR_RANGE = 4,    /* prefill: some |V| > 65280; FP8 / NVFP4 decode: some |q| > 65280
                               (outside fp16); output undefined */
    TA_DEVERR_PAGE = 8      /* paged decode: a block-table entry outside [0, num_pages); output undefined */
};

/*
 * Split-KV plan chosen by the KV-chunk scheduler.  Chunk c of a sequence
 * covers keys [c * chunk, min((c + 1) * chunk, S)).  The decode kernels hand
 * out work items in the order chunk 0 of every (sequence, KV head), chunk 1
 * of every one, and so on.  With up to 128 chunks (and B * Hkv <= 4032) the
 * decode kernel merges the partials itself; otherwise `levels` merge
 * launches of fan-in <= `fanin` follow it (levels = 0 when no merge launch
 * follows).
 */
typedef struct {
    int32_t n_split;        /* chunks per (sequence, KV head)                */
    int32_t chunk;          /* keys per chunk                                */
    int32_t levels;         /* merge launches after the decode kernel        */
    int32_t fanin;          /* partials merged by one warp in one level      */
    int32_t grid;           /* CTAs of the persistent decode kernel          */
    int32_t sm_count;       /* SMs the plan was made for                     */
    size_t workspace_bytes; /* device scratch the call needs                 */
} ta_decode_plan;

/*
 * Full parameter set of a decode call.
 *   q    [B, Hq, D]        in_dtype
 *   k, v [B, Hkv, S, D]    in_dtype (rows at or past seqlens[b] are never read)
 *   out  [B, Hq, D]        out_dtype
 *   lse  [B, Hq]           fp32, may be NULL
 *   seqlens [B] int32 on the device, may be NULL (= every sequence has S keys);
 *     seqlens[b] = 0 gives out = 0 and lse = -inf.  Values outside [0, S]
 *     are clamped on the device and TA_DEVERR_SEQLEN is recorded.
 *   chunk / n_split: 0 = scheduler default; chunk > 0 forces keys per chunk
 *     (takes precedence), else n_split > 0 forces the number of chunks.
 *   wait_limit_ns: every wait of one pipeline stage on another inside the
 *     kernels gives up after this long, records TA_DEVERR_TIMEOUT and ends
 *     the launch (0 = the default of 2 s).  The waits that let a stopping
 *     CTA's own copies and tensor-core operations finish keep the default.
 *   workspace: device scratch of at least ta_decode_plan.workspace_bytes,
 *     256-byte aligned, that the caller zeroes once when it sets it up and
 *     uses for decodes only.  A split decode keeps its status word and one
 *     chunk counter per (sequence, KV head) in the first 16 KiB; every
 *     completed call leaves them zero again (after TA_DEVERR_TIMEOUT, zero
 *     that region again before reuse).
 *     NULL = use the library's own per-device workspace (grown on demand
 *     with cudaMalloc, which synchronises; calls using it on different
 *     streams must not overlap).
 *   With up to 128 chunks (and B * Hkv <= 4032) the decode kernel merges a
 *   sequence's partials itself (the last CTA to finish a chunk of a
 *   (sequence, KV head) merges them); otherwise a separate tree of merge
 *   launches follows it.
 * Supported: D in {64, 128}; in_dtype = out_dtype family F32 or BF16
 * (out may be F32 for BF16 inputs); G in {1, 2, 4} for D = 128 and
 * G in {1, 2, 4, 8} for D = 64.  Pointers q, k, v, out 16-byte aligned.
 */
typedef struct {
    const void *q;
    const void *k;
    const void *v;
    void *out;
    float *lse;
    int32_t B, Hq, Hkv, S, D;
    float scale;
    const int32_t *seqlens;
    ta_dtype in_dtype;
    ta_dtype out_dtype;
    int32_t chunk;
    int32_t n_split;
    void *workspace;
    size_t workspace_bytes;
    void *stream;
    uint64_t wait_limit_ns;  /* time limit of one pipeline wait in the kernels; 0 = 2 s */
} ta_decode_params;

/*
 * Split-KV decode, bf16 q/K/V/out, default plan, library workspace.
 * Exact attention of each of the B*Hq queries over keys [0, L_b) of its KV
 * head, L_b = seqlens[b] or S.  Layouts and rules as in ta_decode_params.
 */
ta_status ta_decode(const void *q, const void *k, const void *v, void *out, float *lse,
                    int B, int Hq, int Hkv, int S, int D, float scale,
                    const int32_t *seqlens, void *stream);

/*
 * Split-KV decode like ta_decode (bf16 q/K/V/out, fp32 lse, default plan),
 * for callers that cannot allocate device memory: it calls no cudaMalloc,
 * cudaFree or other allocating routine.  (The pages this library follows
 * describe no such entry point; it exists for deployment reasons only.)
 * Such callers include programs whose GPU memory is already reserved by a
 * pool allocator (a framework's caching allocator, a serving arena), loops
 * that cannot afford the device-wide synchronisation an allocation can
 * cause, and deployments that forbid allocation after start-up.
 *   Scratch: a fixed 8 MiB array in this library's device code, reserved on
 *   every GPU that loads the library and held until the process exits.  A
 *   shape whose plan needs more (ta_decode_workspace_bytes(B, Hq, Hkv, S, D,
 *   0, 0, seqlens != NULL) > 8 MiB) is rejected with TA_ERR_WORKSPACE and
 *   nothing is launched; such shapes need ta_decode or ta_decode_ex.
 *   Set-up: the first call on each device (or ta_decode_noalloc_setup) has
 *   the CUDA runtime load this library's device code on that device, which
 *   reserves the array there, and looks up its device address with that
 *   device current.  That one-time reservation is the only memory it takes;
 *   make it early: before a pool allocator claims the GPU's memory and
 *   before any stream capture.
 *   Every call clears the scratch's status word and chunk counters on
 *   `stream` before the kernels run.  All calls on one GPU share the one array: calls that may
 *   overlap on the GPU (different streams or host threads with no ordering
 *   between them) race on it and give wrong results.
 *   Device-side flags (TA_DEVERR_*) go to the scratch's status word: read
 *   them with ta_decode_noalloc_status, before the next call clears them.
 *   The per-device address is cached for the life of the process; after a
 *   cudaDeviceReset the next call must not be made on that device.
 * Arguments, layouts, alignment and errors as for ta_decode.
 */
ta_status ta_decode_noalloc(const void *q, const void *k, const void *v, void *out, float *lse,
                            int B, int Hq, int Hkv, int S, int D, float scale,
                            const int32_t *seqlens, void *stream);

/*
 * The one-time set-up of ta_decode_noalloc on the current device, on its
 * own: loads the device code (reserving the fixed scratch array) and looks
 * up the array's address.  Optional; the first ta_decode_noalloc call on a
 * device does the same.  Launches nothing.
 */
ta_status ta_decode_noalloc_setup(void);

/*
 * Read and clear the status word (TA_DEVERR_* bits) of ta_decode_noalloc's
 * fixed scratch on the current device, without allocating: synchronises
 * `stream`, copies the word to the host and zeroes it (and after
 * TA_DEVERR_TIMEOUT the scratch's whole control region).
 */
ta_status ta_decode_noalloc_status(void *stream, int32_t *flags);

/* Split-KV decode with every option of ta_decode_params. */
ta_status ta_decode_ex(const ta_decode_params *p);

/*
 * Split-KV decode over an FP8 (E4M3) KV cache: half the bytes of a bf16
 * cache (the ThriftAttention page, hyperion-consulting.io, "the rise of
 * FP4" and the COMPUTE layer: low-precision KV-cache compression with
 * higher-precision arithmetic).
 *   k, v [B, Hkv, S, D] E4M3 bytes (sign, 4 exponent bits with bias 7, 3
 *   mantissa bits; 0x7f / 0xff are NaN); the cache value of (b, kv head) is
 *   e4m3 * k_scale[b * Hkv + kvh] (resp. v_scale), fp32 on the device, or
 *   1 when the pointer is NULL.  q bf16 (p->in_dtype = TA_BF16), output
 *   bf16 or fp32, fp32 accumulation.  Everything else as ta_decode_ex.
 *   Supported: D = 128, G in {1, 2, 4}.  Queries are used as f16 values
 *   (exact for bf16 values of magnitude in [2^-17, 65280] and zero; below
 *   2^-17 they lose low bits, above 65280 they do not fit, and such a query
 *   records TA_DEVERR_RANGE in the status word, output undefined).
 */
ta_status ta_decode_fp8(const ta_decode_params *p, const float *k_scale, const float *v_scale);

/*
 * Split-KV decode over an NVFP4 KV cache: about a quarter of the bytes of a
 * bf16 cache (the ThriftAttention page, hyperion-consulting.io, "the rise of
 * FP4": NVFP4 KV-cache compression; the COMPUTE layer: low-precision storage
 * inside a kernel that computes in higher precision).
 *   k, v [B, Hkv, S, D/2] bytes: FP4 E2M1 codes (sign, 2 exponent bits with
 *   bias 1, 1 mantissa bit: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), element
 *   2i of a row in the low nibble of byte i, element 2i + 1 in the high one;
 *   k_block_scales, v_block_scales [B, Hkv, S, D/16] bytes: one E4M3 scale per
 *   16 consecutive elements of a row; k_factor, v_factor [B * Hkv] fp32 on
 *   the device, or NULL (1).  The value of element d of key j of (b, kv head)
 *   is e2m1 * e4m3(block d / 16) * factor[b * Hkv + kv head].
 *   q bf16 (p->in_dtype = TA_BF16), output bf16 or fp32, fp32 accumulation;
 *   every element is widened exactly to fp16 on chip, and so is q (as for
 *   ta_decode_fp8, a query element of magnitude above 65280 records
 *   TA_DEVERR_RANGE).  Everything else as ta_decode_ex.
 *   Supported: D = 128, G in {2, 4}, S a multiple of 16, chunks of whole
 *   128-key tiles (the default plan; chunk overrides that are multiples of
 *   128).  k, v, k_block_scales, v_block_scales 16-byte aligned.
 */
ta_status ta_decode_nvfp4(const ta_decode_params *p, const void *k_block_scales, const void *v_block_scales,
                          const float *k_factor, const float *v_factor);

/*
 * Split-KV decode over the key set of pi-Attention (pi-Attention explainer,
 * gist.science/ja/paper/2511.10696, technical summary section 2A): the
 * query of each sequence, the newest token i = L_b - 1, attends
 *   the ring-local window  { j : max(0, i - window) <= j <= i }  and
 *   the periodic skips     { j = i - m * period : m >= 1, 0 <= j < i - window },
 * in one softmax (causal: past keys only).  The learned fusion gate of that
 * page is not applied (it needs trained weights): every attended key has
 * its plain score.  period = 1 attends every key (= ta_decode_ex).
 *   Arguments as ta_decode_ex (K/V contiguous [B, Hkv, S, D]); window >= 0,
 *   period >= 1.  The chunks cut the ascending list of attended keys: a
 *   caller workspace needs ta_decode_pi_workspace_bytes(...) bytes.
 */
ta_status ta_decode_pi(const ta_decode_params *p, int window, int period);

/* Workspace bytes of ta_decode_pi (0 on bad arguments); arguments as
 * ta_decode_workspace_bytes plus window and period. */
size_t ta_decode_pi_workspace_bytes(int B, int Hq, int Hkv, int S, int D, int chunk, int n_split, int varlen,
                                    int window, int period);

/*
 * Split-KV decode over a paged KV cache (block table).  The step beside the
 * variable-length batch: the KV cache is a pool of fixed-size pages and each
 * sequence lists its pages, so sequences grow without copying (Attention
 * glossary, jisaku.com/glossary/attention, "the memory bandwidth and VRAM
 * wall": the KV cache dominates decode memory).  Same result as ta_decode_ex
 * on the gathered contiguous cache.
 *   k_pages, v_pages [num_pages, Hkv, page_size, D] (head-major inside a
 *     page, so one head's rows of a page are contiguous), in_dtype;
 *   block_table [B, pages_per_seq] int32 on the device: key j of sequence b
 *     is row j % page_size of page block_table[b][j / page_size];
 *   seqlens [B] int32 on the device, required; 0 <= seqlens[b] <=
 *     pages_per_seq * page_size (else clamped, TA_DEVERR_SEQLEN).  Entries
 *     beyond a sequence's last page are never read.  A page id outside
 *     [0, num_pages) is not followed: TA_DEVERR_PAGE is recorded and the
 *     output is undefined.
 *   q, out, lse, dtypes, chunk / n_split and workspace as in
 *   ta_decode_params, with S = pages_per_seq * page_size (the plan and
 *   workspace are those of ta_decode_plan_for(B, Hq, Hkv, S, D, chunk,
 *   n_split, 1, 0, ...)).  k_pages, v_pages 16-byte aligned.
 */
typedef struct {
    const void *q;
    const void *k_pages;
    const void *v_pages;
    const int32_t *block_table;
    const int32_t *seqlens;
    void *out;
    float *lse;
    int32_t B, Hq, Hkv, D;
    int32_t page_size, pages_per_seq, num_pages;
    float scale;
    ta_dtype in_dtype;
    ta_dtype out_dtype;
    int32_t chunk;
    int32_t n_split;
    void *workspace;
    size_t workspace_bytes;
    void *stream;
    uint64_t wait_limit_ns;  /* as in ta_decode_params; 0 = 2 s */
} ta_paged_decode_params;

ta_status ta_decode_paged(const ta_paged_decode_params *p);

/*
 * The split phase alone: every (sequence b, query head h, chunk c) partial
 * of ta_decode_ex, written to caller buffers and not merged.
 *   m, l [B*Hq, n_split] fp32, o [B*Hq, n_split, D] fp32, row r = b*Hq + h,
 *   with n_split the plan's (ta_decode_plan_for with the same chunk /
 *   n_split / seqlens choice).  m is in natural-log units; an empty chunk
 *   gives m = -inf, l = 0, o = 0.  Merging them with ta_combine gives the
 *   decode result.  p->out and p->lse are ignored; p->workspace may be NULL
 *   or any zeroed 256-byte-aligned buffer of >= 256 bytes (only its status
 *   word is used).  o 16-byte aligned; m, l 4-byte aligned.
 */
ta_status ta_decode_partials(const ta_decode_params *p, float *m, float *l, float *o);

/*
 * The plan ta_decode_ex would use (pure host computation; launches nothing).
 * varlen != 0 when seqlens will be passed (the chunking then
 * over-decomposes, since lengths are only known on the device).
 * sm_count = 0 queries the current device.  chunk / n_split as in
 * ta_decode_params.
 */
ta_status ta_decode_plan_for(int B, int Hq, int Hkv, int S, int D, int chunk, int n_split, int varlen,
                             int sm_count, ta_decode_plan *plan);

/* Workspace bytes of ta_decode_plan_for(...) on the current device (0 on error). */
size_t ta_decode_workspace_bytes(int B, int Hq, int Hkv, int S, int D, int chunk, int n_split,
                                 int varlen);

/*
 * Read and clear the device status word (TA_DEVERR_* bits) of a decode
 * workspace (NULL = the library's own workspace of the current device; if
 * TA_DEVERR_TIMEOUT is set its whole 16 KiB control region is cleared too).
 * Synchronises `stream` first.
 */
ta_status ta_decode_status(void *workspace, void *stream, int32_t *flags);

/*
 * Log-sum-exp merge of N split-KV partials for each of R rows (the tree
 * combine of the Tree Attention explainer, sections 1 and 3, on one GPU):
 *   m, l [R, N] fp32 (m natural-log units; any finite reference point, or
 *   -inf with l = 0 for an empty partial), o [R, N, D] fp32 unnormalised.
 *   m* = max_i m_i, l* = sum_i l_i e^(m_i - m*), o* = sum_i o_i e^(m_i - m*)
 *   out [R, D] (out_dtype) = o* / l*;  lse [R] = m* + ln l* (may be NULL).
 *   A row whose partials are all empty gives out = 0, lse = -inf.
 * Fan-in <= 64 is one warp per row; larger N merges in levels of 64, with
 * intermediates in `workspace` (>= ta_combine_workspace_bytes(R, N, D);
 * NULL = library workspace).  D in {64, 128}; R >= 1; N >= 1.
 */
ta_status ta_combine(const float *m, const float *l, const float *o, int R, int N, int D,
                     void *out, ta_dtype out_dtype, float *lse,
                     void *workspace, size_t workspace_bytes, void *stream);

/* Scratch bytes ta_combine needs for (R, N, D); 0 when no level writes intermediates. */
size_t ta_combine_workspace_bytes(int R, int N, int D);

/*
 * Causal prefill, fused QK^T * scale -> softmax -> PV on the tensor cores
 * (the fusion of matmul, scaling and softmax that the Grayskull SRAM
 * attention explainer, aibr.jp/archives/146339, section 3, describes),
 * bf16 in and out, fp32 accumulation.
 *   q, out [B, H, S, D] bf16; k, v [B, Hkv, S, D] bf16; lse [B, H, S] fp32
 *   (may be NULL).  Query row i attends keys 0..i (top-left aligned, square).
 * The softmax weights P enter the PV product as fp16 (relative rounding
 * 2^-12), with V converted to fp16 on chip; |V| must be <= 65280.  The row
 * sums l are taken over the same fp16 weights.
 * Supported: D = 128; H % Hkv == 0; S >= 1; scale > 0; q, k, v, out
 * 16-byte aligned.  The library's status word (read with
 * ta_decode_status(NULL, ...)) records TA_DEVERR_TIMEOUT if a pipeline wait
 * gave up and TA_DEVERR_RANGE if some |V| exceeded the fp16 range.
 */
ta_status ta_prefill_causal(const void *q, const void *k, const void *v, void *out, float *lse,
                            int B, int H, int Hkv, int S, int D, float scale, void *stream);

/*
 * Causal prefill with every option: the batched layouts of
 * ta_prefill_causal, or (cu_seqlens != NULL) the packed layouts of
 * ta_prefill_causal_varlen, with the output in bf16 or fp32.
 *   q, k, v, out, lse, H, Hkv, D, scale: as ta_prefill_causal (batched) or
 *     ta_prefill_causal_varlen (packed);
 *   batched: B sequences of S tokens, cu_seqlens = NULL, total_tokens unused;
 *   packed:  B = number of sequences, S = max_seqlen, cu_seqlens [B + 1] and
 *     total_tokens as ta_prefill_causal_varlen;
 *   out_dtype: TA_BF16 (out rounded to nearest even) or TA_F32 (the fp32
 *     value the bf16 output is rounded from; same kernel, same arithmetic);
 *   wait_limit_ns: as in ta_decode_params (0 = 2 s).
 * Errors and device-side flags as ta_prefill_causal.
 */
typedef struct {
    const void *q;
    const void *k;
    const void *v;
    void *out;
    float *lse;
    int32_t B, H, Hkv, S, D;
    float scale;
    const int32_t *cu_seqlens;
    int32_t total_tokens;
    ta_dtype out_dtype;
    uint64_t wait_limit_ns;
    void *stream;
} ta_prefill_params;

ta_status ta_prefill_causal_ex(const ta_prefill_params *p);

/*
 * Causal prefill of a packed batch of variable-length sequences: the
 * prefill-side twin of the variable-length decode, same fused kernel.
 * Sequence s is tokens [cu_seqlens[s], cu_seqlens[s+1]) of the packed
 * tensors; within it query row i attends keys 0..i of the same sequence.
 *   q, out [total_tokens, H, D] bf16; k, v [total_tokens, Hkv, D] bf16;
 *   lse [H, total_tokens] fp32 (may be NULL);
 *   cu_seqlens [num_seqs + 1] int32 on the device, non-decreasing, from 0 to
 *     total_tokens; every sequence at most max_seqlen tokens long.  Offsets
 *     that break this are not followed past the tensors:
 *     TA_DEVERR_SEQLEN is recorded (read with ta_decode_status(NULL, ...))
 *     and rows past max_seqlen are not written.
 * Keys of a neighbouring sequence that share a 128-key tile with attended
 * keys are masked (weight exactly 0), so they must be finite.
 * Supported: D = 128; H % Hkv == 0; scale > 0; q, k, v, out 16-byte aligned.
 */
ta_status ta_prefill_causal_varlen(const void *q, const void *k, const void *v, void *out, float *lse,
                                   const int32_t *cu_seqlens, int num_seqs, int max_seqlen, int total_tokens,
                                   int H, int Hkv, int D, float scale, void *stream);

/*
 * Test hook: the next `count` kernel launches of this process (any entry
 * point, any thread) are not made; the call that would make each returns
 * TA_ERR_CUDA with a message naming this hook, after its argument checks and
 * before anything further is enqueued.  count = 0 cancels.  Returns the
 * number that was pending.  For testing callers' error handling; a launch
 * that is not made computes nothing and writes no output.
 */
int ta_test_fail_next_launches(int count);

/*
 * Test hook for the device-side time limit: in each of the next `count`
 * kernel launches that have pipeline waits (decode and prefill kernels, not
 * the merge), the CTAs' producer first waits on a barrier that nothing
 * completes, so that wait runs out after the launch's wait_limit_ns: the
 * launch then stops every role, lets what it issued finish, frees its tensor
 * memory, records TA_DEVERR_TIMEOUT and returns; its outputs are not
 * written.  count = 0 cancels.  Returns the number that was pending.
 */
int ta_test_stall_next_launches(int count);

/* Message for the calling thread's last non-OK status ("" if none). */
const char *ta_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* TA_H */
