/*
 * ffd.h -- C ABI of libffd.so: Faster Flash Decoding (FFD) sparse decode attention on one
 * NVIDIA GB300 (sm_103a).
 *
 * Method source: "Faster Than Flash: Exploiting Attention Sparsity for Efficient Long-Context
 * Decoding" (technical summary pages), Methodology §1 "Content-aware scanning via low-bit
 * quantization", §2 "Top-delta selection strategy", §3 "Fused kernel and system optimisation".
 * The pages call FFD a drop-in replacement for a standard attention kernel (Significance §2),
 * so the decode entry point has the shape of a paged flash-decode call.
 *
 * Conventions for every function:
 *   - Pointers marked "device" are device memory owned by the caller; the library allocates no
 *     memory and keeps no state between calls other than what the caller's workspace holds.
 *     One exception: ffd_decode_attention_static keeps its scratch in a static device array of
 *     the library (and that array's address per device); see its own comment.
 *   - Calls are asynchronous on the given stream (a cudaStream_t passed as void*; NULL is the
 *     legacy default stream), except ffd_get_error, which synchronises that stream.
 *   - Argument errors are detected on the host before anything is enqueued and returned as a
 *     status. Launch failures return FFD_ERR_CUDA. Problems only the device can see (a block
 *     table entry out of range, a key outside the fp16 range) set bits in a device error word
 *     and are read with ffd_get_error; the kernels never trap.
 *   - Supported shapes: head_dim = 128, page_size = 64, 1 <= num_q_heads/num_kv_heads <= 8.
 *     Anything else returns FFD_ERR_UNSUPPORTED.
 *
 * Paged cache layout (P pages, Hkv KV heads, 64 tokens per page, d = 128 channels, channel
 * group g = c/32 of channel c, token r = 0..63 of a page):
 *   K, V    bf16 [P][Hkv][64][128]
 *   thumb   u8   [P][Hkv][FFD_THUMB_RECORD_BYTES]  one thumbnail record per (page, KV head):
 *             bytes [0, 2048)     2-bit codes: token r at 32 r, channel c in byte c/4, bits
 *                                 2(c%4)+{0,1}
 *             bytes [2048, 2560)  f16 thumbnail scale of token r, group g at 2048 + 8 r + 2 g
 *             bytes [2560, 3072)  f16 thumbnail zero (offset), at 2560 + 8 r + 2 g
 *   resid   u8   [P][Hkv][FFD_RESID_RECORD_BYTES]  one residual record per (page, KV head):
 *             bytes [0, 8192)     int8 residual codes: token r at 128 r; the 16-byte chunk j of
 *                                 a token (channels 16j .. 16j+15, in order) is stored at chunk
 *                                 position j ^ (r % 8), i.e. channel c at
 *                                 128 r + 16 ((c / 16) ^ (r % 8)) + c % 16
 *             bytes [8192, 8704)  f16 residual scale of token r, group g at 8192 + 8 r + 2 g
 * Each record is what one stage of the method reads for a block, so a kernel moves it with one
 * bulk copy; the chunk permutation of the residual codes is the order in which the decode kernel
 * reads them from shared memory without bank conflicts.
 * Logical block b of sequence s (tokens 64b .. 64b+63) lives in page block_table[s][b].
 */
#ifndef FFD_H
#define FFD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FFD_OK = 0,
    FFD_ERR_INVALID_ARG = 1, /* null pointer, negative size, inconsistent shape */
    FFD_ERR_UNSUPPORTED = 2, /* head_dim != 128, page_size != 64, GQA group size outside 1..8 */
    FFD_ERR_WORKSPACE = 3,   /* workspace smaller than the matching *_workspace_size() */
    FFD_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
    FFD_ERR_BOUNDS = 5,      /* device: a block_table / page_ids entry outside [0, num_pages) */
    FFD_ERR_RANGE = 6,       /* device: a key outside the fp16 range (|k| >= 65504 or NaN), or a
                                query with |q| >= 2^27 */
    FFD_ERR_TIMEOUT = 7,     /* device: a pipeline wait exceeded its bound (params wait_limit_us,
                                2 s by default); the call's results are invalid */
} ffd_status;

#define FFD_THUMB_RECORD_BYTES 3072
#define FFD_RESID_RECORD_BYTES 8704

/* Bits of the device error word (first 4 bytes of a workspace, or the quantiser's word). */
#define FFD_ERRBIT_BOUNDS 0x1
#define FFD_ERRBIT_RANGE 0x2
#define FFD_ERRBIT_TIMEOUT 0x4

/* Static description of a paged key/value cache. */
typedef struct {
    int32_t num_pages;    /* P >= 1 */
    int32_t num_kv_heads; /* Hkv >= 1 */
    int32_t head_dim;     /* must be 128 */
    int32_t page_size;    /* must be 64 */
} ffd_cache_desc;

/* One decode step: every sequence contributes one query token with num_q_heads heads. */
typedef struct {
    int32_t batch;              /* B >= 1 sequences */
    int32_t num_q_heads;        /* Hq, a multiple of num_kv_heads */
    int32_t num_kv_heads;       /* Hkv; G = Hq / Hkv query heads share a KV head (GQA) */
    int32_t head_dim;           /* must be 128 */
    int32_t page_size;          /* must be 64 */
    int32_t num_pages;          /* P, bound for block_table entries */
    int32_t max_blocks_per_seq; /* row stride of block_table; seq_lens[b] <= 64 * this */
    int32_t sink_tokens;        /* S >= 0: tokens 0 .. S-1 are sink tokens */
    int32_t local_tokens;       /* L >= 0: tokens n-L .. n-1 are local tokens */
    float delta;                /* delta of the Top-delta rule; +INFINITY keeps every block */
    float sm_scale;             /* score scale, finite and > 0; normally 1/sqrt(head_dim) */
    int32_t num_splits;         /* 0: library's choice (one per SM, or one per 4 blocks of
                                   batch * num_kv_heads * max_blocks_per_seq when that is
                                   fewer); else the number of KV partitions, i.e. the CTAs of
                                   the persistent kernel of ffd_decode_attention or
                                   ffd_dense_decode, at most one per SM: larger values are
                                   clamped to the SM count */
    int32_t wait_limit_us;      /* >= 0. Bound, in microseconds, of every wait inside a kernel of
                                   this call (a CTA waiting for a copy, for another warp or for
                                   another CTA); 0 takes the default of 2 s. A wait that runs out
                                   sets FFD_ERRBIT_TIMEOUT, the CTA stops waiting and drains its
                                   own copies, and the kernel ends (results invalid). */
    int32_t schedule;           /* the order of the work of ffd_decode_attention(_static), with
                                   the same results: FFD_SCHEDULE_FUSED (0) or
                                   FFD_SCHEDULE_SCAN_REFINE (1), below; ignored by the masked,
                                   dense, selector and ART calls */
} ffd_decode_params;

/* Schedules of the decode step (ffd_decode_params.schedule). Both compute the same step.
 *   FFD_SCHEDULE_FUSED: one pipeline per CTA over an equal share of all blocks; the scan of a
 *     block's thumbnail and the refinement of the kept blocks before it overlap. Suits steps that
 *     keep most blocks (the refinement's bytes dominate).
 *   FFD_SCHEDULE_SCAN_REFINE: every CTA first scans an equal share of all thumbnails with all its
 *     compute warps, then, after a grid-wide barrier, the kept blocks of all CTAs are shared out
 *     equally for the refinement. Suits steps that drop most blocks (the scan dominates, and the
 *     kept blocks may crowd into a few sequences). A caller can pick it from the kept fraction of
 *     the previous step (keep_mask). It needs batch * num_kv_heads * max_blocks_per_seq <=
 *     INT32_MAX (else FFD_ERR_UNSUPPORTED). */
#define FFD_SCHEDULE_FUSED 0
#define FFD_SCHEDULE_SCAN_REFINE 1

/* The schedule this library suggests for a step over total_blocks blocks (sum over sequences and
 * KV heads of ceil(n / 64)) when the previous step kept kept_blocks of them (the count of ones in
 * its keep_mask): FFD_SCHEDULE_SCAN_REFINE when fewer than half the blocks were kept and there are
 * at least 64 blocks per SM of the current device, else FFD_SCHEDULE_FUSED (also for arguments
 * out of range). Host only; reads the device's SM count once. */
int32_t ffd_suggest_schedule(int64_t total_blocks, int64_t kept_blocks);

/* Human-readable name of a status. Never NULL. */
const char *ffd_status_string(ffd_status status);

/* The cudaError_t behind the latest FFD_ERR_CUDA returned on the calling thread (0 if none
 * yet); kept per thread until the next such failure. */
int32_t ffd_last_cuda_error(void);

/* Library version, major * 10000 + minor * 100 + patch (3.00: ffd_decode_params gained
 * wait_limit_us and schedule). */
int32_t ffd_version(void);

/*
 * ffd_quantize_keys -- split bf16 keys into the 2-bit thumbnail and the int8 residual.
 * Source: Methodology §1 (the K cache is partitioned into 2-bit quantized thumbnails used to
 * estimate attention scores and 8-bit residuals that rebuild the keys close to fp16 precision).
 * Format (the pages leave it open; fixed by this library), per token, KV head and group g of 32
 * channels, all steps single-rounded IEEE fp32:
 *   zero = f16(min x), scale = f16((max x - min x) / 3),
 *   c2 = clamp(rint((x - zero) / scale), 0, 3)  (0 if scale == 0),
 *   r = x - fma(c2, scale, zero), r_scale = f16(max |r| / 127),
 *   c8 = clamp(rint(r / r_scale), -127, 127)     (0 if r_scale == 0);
 * rint rounds half to even; a signed zero minimum or maximum counts as +0.
 *
 *   cache         shape of the cache (head_dim 128, page_size 64)
 *   k_bf16        device, bf16 [P][Hkv][64][128], read only
 *   thumb, resid  device outputs, the records above (written for the selected pages only),
 *                 16-byte aligned
 *   page_ids      device int32 [num_page_ids] pages to quantise, or NULL for all P pages
 *   num_page_ids  number of entries in page_ids (ignored when page_ids is NULL)
 *   error_word    device int32, or NULL: FFD_ERRBIT_BOUNDS is OR-ed in for a page id outside
 *                 [0, P) (that page is skipped), FFD_ERRBIT_RANGE for a key with |k| >= 65504 or
 *                 NaN (its group is still written; its contents are then unspecified)
 *   stream        cudaStream_t
 * Returns FFD_OK, FFD_ERR_INVALID_ARG, FFD_ERR_UNSUPPORTED or FFD_ERR_CUDA.
 */
ffd_status ffd_quantize_keys(const ffd_cache_desc *cache, const void *k_bf16, uint8_t *thumb,
                             uint8_t *resid, const int32_t *page_ids, int32_t num_page_ids,
                             int32_t *error_word, void *stream);

/*
 * ffd_append_kv -- append one new token per sequence to the paged cache: quantise its key into
 * the thumbnail and residual records and store its value (and, optionally, the raw key).
 * Source: Methodology §1 (the K cache is kept as 2-bit thumbnails plus 8-bit residuals); in a
 * decode loop every generated token is added to that cache before the next attention step, so
 * this is the incremental form of ffd_quantize_keys. The token's codes and scales are bit for
 * bit those ffd_quantize_keys writes for the same key.
 *
 *   cache        shape of the cache (head_dim 128, page_size 64)
 *   batch        B >= 1 sequences
 *   max_blocks_per_seq  row stride of block_table (>= 1)
 *   k_new_bf16   device bf16 [B][Hkv][128], the new keys, 16-byte aligned
 *   v_new_bf16   device bf16 [B][Hkv][128], the new values, 16-byte aligned
 *   positions    device int32 [B]: token index p of the new token of sequence b (normally its
 *                length before the append); it is stored in row p % 64 of page
 *                block_table[b][p / 64]. A negative entry appends nothing for that sequence.
 *   block_table  device int32 [B][max_blocks_per_seq]
 *   thumb, resid device records (layout above): the token's row is rewritten, nothing else
 *   v_bf16       device bf16 [P][Hkv][64][128]: the token's row receives the new value
 *   k_bf16       device bf16 [P][Hkv][64][128] or NULL: the token's row receives the raw key
 *   error_word   device int32, or NULL: FFD_ERRBIT_BOUNDS for p >= 64 * max_blocks_per_seq or a
 *                page outside [0, P) (that sequence is skipped), FFD_ERRBIT_RANGE for a key
 *                outside the fp16 range (written as by ffd_quantize_keys)
 *   stream       cudaStream_t
 * Two sequences that name the same (page, row) race; the caller's block table must not do that.
 * Returns FFD_OK, FFD_ERR_INVALID_ARG, FFD_ERR_UNSUPPORTED or FFD_ERR_CUDA.
 */
ffd_status ffd_append_kv(const ffd_cache_desc *cache, int32_t batch, int32_t max_blocks_per_seq,
                         const void *k_new_bf16, const void *v_new_bf16, const int32_t *positions,
                         const int32_t *block_table, uint8_t *thumb, uint8_t *resid,
                         void *v_bf16, void *k_bf16, int32_t *error_word, void *stream);

/*
 * Bytes of device workspace that ffd_decode_attention needs for these parameters on the current
 * device. Returns 0 for parameters that ffd_decode_attention would reject.
 */
size_t ffd_decode_workspace_size(const ffd_decode_params *params);

/*
 * ffd_decode_attention -- one FFD decode-attention step.
 * Source: Methodology §2 (keep token j when s_ij >= m~_i - delta, m~_i a pseudo-max taken over
 * the sink and local tokens only) and §3 (stage 1 pseudo-max estimation from sink and local
 * tokens; stage 2 streams the 2-bit keys, computes provisional scores and filters blocks against
 * the threshold; stage 3 loads the 8-bit residuals and V of the selected blocks and computes
 * exact attention). Per sequence b (length n = seq_lens[b]) and query head i of KV head h:
 *   K^_j = fma(c8, r_scale, fma(c2, scale, zero)) (thumbnail + residual), x^_j = thumbnail only,
 *   s_ij = sm_scale * q_i . K^_j,  s^_ij = sm_scale * q_i . x^_j,
 *   m~_i = max of s_ij over j < S and n-L <= j < n,
 *   block c (tokens 64c .. 64c+63, j < n) is kept when it holds a sink or local token, or when
 *   some head i of the group and token j of the block give s^_ij >= m~_i - delta,
 *   out_i = softmax over the kept tokens of s_ij, applied to V (dropped tokens contribute 0).
 * n = 0 gives out_i = 0 and m~_i = -inf. S = L = 0 gives m~ = -inf, so every block is kept.
 *
 *   q_bf16      device bf16 [B][Hq][128], |q| < 2^27 (else FFD_ERRBIT_RANGE)
 *   thumb, resid, v_bf16   device cache in the layout above (records from ffd_quantize_keys),
 *               16-byte aligned. Rows of a sequence's last page at or past n are never used:
 *               they may hold any bits (their V rows are zeroed on chip before P.V).
 *   seq_lens    device int32 [B], 0 <= seq_lens[b] <= 64 * max_blocks_per_seq
 *   block_table device int32 [B][max_blocks_per_seq]; only entries b < ceil(n/64) are read
 *   out         device fp32 [B][Hq][128]
 *   keep_mask   device u8 [B][Hkv][max_blocks_per_seq] or NULL: 1 = block kept, 0 = dropped;
 *               entries at or past ceil(n/64) are set to 0
 *   m_tilde     device fp32 [B][Hq] or NULL: the pseudo-max
 *   workspace   device, >= ffd_decode_workspace_size(params) bytes, 256-byte aligned. Its
 *               first 4 bytes are the device error word. Zero-fill it once before first use;
 *               each call leaves it ready for the next one (zero-fill it again after a call that
 *               reported FFD_ERR_TIMEOUT). Calls that share a workspace must be ordered on one
 *               stream.
 * Launch: one cooperative kernel of at most one CTA per SM whose CTAs exchange the stage-1
 * maxima, so all of them must be resident at once; a launch that cannot be (SMs held by other
 * work under an SM limit) fails with FFD_ERR_CUDA and enqueues nothing.
 * Errors: host-side status as listed above; FFD_ERRBIT_BOUNDS in the workspace error word when
 * a block_table entry lies outside [0, num_pages) (the block is treated as empty).
 */
ffd_status ffd_decode_attention(const ffd_decode_params *params, const void *q_bf16,
                                const uint8_t *thumb, const uint8_t *resid, const void *v_bf16,
                                const int32_t *seq_lens, const int32_t *block_table, float *out,
                                uint8_t *keep_mask, float *m_tilde, void *workspace,
                                size_t workspace_bytes, void *stream);

/* Bytes of device workspace that ffd_dense_decode needs (same rules as above). */
size_t ffd_dense_workspace_size(const ffd_decode_params *params);

/*
 * ffd_dense_decode -- dense bf16 flash-decode attention, the in-library comparison kernel:
 * out_i = softmax_j(sm_scale * q_i . K_j) V over every token j < n, with the original bf16 keys.
 * Source: the pages compare FFD against FlashAttention-2 decoding (Main results, kernel speedup
 * and end-to-end throughput). sink_tokens, local_tokens and delta are ignored.
 *   k_bf16, v_bf16  device bf16 [P][Hkv][64][128]; other arguments as in ffd_decode_attention
 *   (the workspace rules and the cooperative launch included).
 */
ffd_status ffd_dense_decode(const ffd_decode_params *params, const void *q_bf16,
                            const void *k_bf16, const void *v_bf16, const int32_t *seq_lens,
                            const int32_t *block_table, float *out, void *workspace,
                            size_t workspace_bytes, void *stream);

/* Comparison selectors of ffd_select_blocks. */
#define FFD_SELECT_TOPK 1
#define FFD_SELECT_TOPP 2

/*
 * Bytes of device workspace that ffd_select_blocks needs for these parameters (0 for parameters
 * it would reject, including max_blocks_per_seq > 16384).
 */
size_t ffd_select_workspace_size(const ffd_decode_params *params);

/*
 * ffd_select_blocks -- choose blocks by one of the comparison rules the method is measured
 * against: fixed-budget Top-k or distribution-adaptive Top-p on the same thumbnail scores.
 * Source: Problem statement (the selection dilemma: Top-k does not adapt to attention entropy;
 * Top-p needs a global softmax and a sort). The pages give no detailed definition; this library's:
 *   s^_ij = sm_scale * q_i . x^2_j (thumbnail only, as in stage 2 of ffd_decode_attention);
 *   Top-k (selector FFD_SELECT_TOPK, budget = k, a non-negative integer): importance of block c =
 *     max over the group's heads i and its tokens j < n of s^_ij; the k non-forced blocks of
 *     largest importance are kept (ties: lower block index first);
 *   Top-p (FFD_SELECT_TOPP, budget = p in (0, 1]): per head i, P_ij = softmax over all j < n of
 *     s^_ij and block mass m_ic = sum of P_ij over the block; blocks ranked by mass (descending,
 *     ties: lower index first) are kept while the masses ranked before them sum to less than p
 *     (the shortest prefix reaching p); the union over the group's heads is kept.
 * Both keep the blocks holding a sink or local token, like ffd_decode_attention.
 *   params      as for ffd_decode_attention (delta is ignored)
 *   q_bf16, thumb, seq_lens, block_table   as for ffd_decode_attention
 *   keep_mask   device u8 [B][Hkv][max_blocks_per_seq] output: 1 = kept; entries at or past
 *               ceil(n/64) are set to 0
 *   workspace   device, >= ffd_select_workspace_size(params) bytes, 256-byte aligned; its first
 *               4 bytes are the device error word (zero it before first use)
 * Two kernel launches (a pass over every thumbnail, then one CTA per (sequence, KV head) that
 * sorts its blocks). Errors: as ffd_decode_attention; FFD_ERR_INVALID_ARG for a bad selector or
 * budget; FFD_ERRBIT_BOUNDS for a block-table entry outside [0, P) (that block scores -inf).
 */
ffd_status ffd_select_blocks(const ffd_decode_params *params, int32_t selector, float budget,
                             const void *q_bf16, const uint8_t *thumb, const int32_t *seq_lens,
                             const int32_t *block_table, uint8_t *keep_mask, void *workspace,
                             size_t workspace_bytes, void *stream);

/*
 * ffd_decode_attention_masked -- stage 3 of the decode step over a caller-given block mask (for
 * instance one from ffd_select_blocks): out_i = softmax over the tokens j < n of the given blocks
 * of s_ij = sm_scale * q_i . K^_j, applied to V (the exact scores of ffd_decode_attention).
 * Source: Methodology §3 (stage 3: exact attention over the selected blocks).
 *   keep_in     device u8 [B][Hkv][max_blocks_per_seq]: nonzero = attend to the block. The mask
 *               alone decides: sink and local blocks are not added.
 *   keep_mask   device u8 [B][Hkv][max_blocks_per_seq] or NULL: the mask used (keep_in less the
 *               blocks whose block-table entry is out of range)
 *   other arguments, workspace rules and errors as ffd_decode_attention (delta is ignored;
 *   m_tilde still reports the pseudo-max of the sink and local tokens).
 */
ffd_status ffd_decode_attention_masked(const ffd_decode_params *params, const void *q_bf16,
                                       const uint8_t *thumb, const uint8_t *resid,
                                       const void *v_bf16, const int32_t *seq_lens,
                                       const int32_t *block_table, const uint8_t *keep_in,
                                       float *out, uint8_t *keep_mask, float *m_tilde,
                                       void *workspace, size_t workspace_bytes, void *stream);

/*
 * ffd_art_attention -- attention with run-time termination (ART) over the blocks of a mask:
 * each (sequence, KV head) unit walks block 0, then the blocks of keep_in (or all blocks) from the
 * most recent to the oldest, folding each into an online softmax, and stops early once its
 * partial output is stable.
 * Source: "ART: Attention Run-time Termination" (technical summary page), §2.2 (stop when the
 * change in magnitude and the change in direction of the partial output both fall below tau and
 * phi), §2.3 (the criterion must hold `patience` times in a row), §2.4 (any block order is exact
 * because online softmax is permutation invariant; block 0 is always evaluated first). The FFD
 * pages name ART as an orthogonal layer. This library's reading: after t >= 2 blocks, with
 * P_i(t) = o_i / l_i the normalised partial output of head i,
 *   d_scale = max_i | |P_i(t)| - |P_i(t-1)| | / |P_i(t-1)|,
 *   d_direction = max_i (1 - cos(P_i(t), P_i(t-1))) over the group's heads,
 * the criterion is d_scale < tau and d_direction < phi (strict), and the unit stops after the
 * block at which it has held `patience` times in a row. Scores are the exact
 * s_ij = sm_scale * q_i . K^_j of ffd_decode_attention.
 *   params      as for ffd_decode_attention (delta, sink_tokens, local_tokens and num_splits are
 *               ignored)
 *   tau, phi    thresholds, >= 0 (0 disables termination: every listed block is used)
 *   patience    >= 1
 *   q_bf16, thumb, resid, v_bf16, seq_lens, block_table   as for ffd_decode_attention
 *   keep_in     device u8 [B][Hkv][max_blocks_per_seq] or NULL (all blocks): nonzero = the block
 *               may be visited; block 0 is visited whatever it says
 *   out         device f32 [B][Hq][128]: o / l after the last block used (0 for n = 0)
 *   blocks_used device i32 [B][Hkv] or NULL: blocks folded in per unit
 *   workspace   device, >= ffd_art_workspace_size(params) bytes, 256-byte aligned; its first 4
 *               bytes are the device error word (zero it before first use), then one traversal
 *               list of max_blocks_per_seq int32 per (sequence, KV head), rewritten every call
 * One kernel launch, one CTA per (sequence, KV head): the traversal of a unit is sequential
 * through the probe, so three groups of the CTA score the next blocks into per-block states while
 * four warps merge them in order, two blocks at a time, and take the probes; the parallelism
 * beyond that is across units. Errors: FFD_ERR_INVALID_ARG for NULL pointers, misaligned
 * buffers, tau or phi negative or NaN, patience < 1; otherwise as ffd_decode_attention
 * (FFD_ERRBIT_BOUNDS for a block-table entry outside [0, P): that block contributes nothing).
 */
size_t ffd_art_workspace_size(const ffd_decode_params *params);
ffd_status ffd_art_attention(const ffd_decode_params *params, float tau, float phi,
                             int32_t patience, const void *q_bf16, const uint8_t *thumb,
                             const uint8_t *resid, const void *v_bf16, const int32_t *seq_lens,
                             const int32_t *block_table, const uint8_t *keep_in, float *out,
                             int32_t *blocks_used, void *workspace, size_t workspace_bytes,
                             void *stream);

/*
 * ffd_decode_attention_static -- ffd_decode_attention without a caller-supplied workspace.
 * The paper has no counterpart: this entry point exists for callers that cannot allocate device
 * memory for a workspace, such as a plain C host that links only this library and owns no device
 * allocator, or a serving process that has committed all device memory to its KV-cache pool and
 * must not allocate (or synchronise the device through cudaMalloc) inside its decode loop.
 *
 * It computes exactly what ffd_decode_attention computes, with the same arguments minus the
 * workspace. Its scratch (stage-1 maxima, split records, counters) is a static device array
 * of 4 MiB inside libffd.so, held by every GPU that loads the library until the process exits.
 * Nothing is allocated and no allocating routine is called.
 *   - Limit: parameters whose ffd_decode_workspace_size() exceeds 4 MiB are rejected with
 *     FFD_ERR_WORKSPACE before anything is enqueued (use ffd_decode_attention for those).
 *   - Set-up: the first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current, and looks it up again whenever the
 *     thread's current CUDA context is not the one of the last look-up (a cudaDeviceReset
 *     replaces the primary context and the array's address with it); make the first call after
 *     such a change before any stream capture. A failed look-up returns FFD_ERR_CUDA.
 *   - Sharing: every call on a device uses the same array and it keeps the previous call's
 *     contents; each call clears the parts that must start at zero (error word, merge tickets,
 *     slot counters)
 *     on its stream. Calls whose executions overlap on the GPU race with each other: order them
 *     on one stream (or with events).
 *   - error_word: device int32 or NULL. Device-detected errors (FFD_ERRBIT_*) are OR-ed into it;
 *     read and clear it with ffd_get_error. With NULL they are not reported.
 */
ffd_status ffd_decode_attention_static(const ffd_decode_params *params, const void *q_bf16,
                                       const uint8_t *thumb, const uint8_t *resid,
                                       const void *v_bf16, const int32_t *seq_lens,
                                       const int32_t *block_table, float *out,
                                       uint8_t *keep_mask, float *m_tilde, int32_t *error_word,
                                       void *stream);

/*
 * ffd_set_profile_events -- optional instrumentation. While both events are non-NULL, every
 * ffd_decode_attention / ffd_dense_decode call records `start` on its stream right before its
 * main kernel (the fused stage-1/2/3 kernel, or the dense kernel) and `stop` right after it, so the
 * caller can time that kernel alone with cudaEventElapsedTime. The events are cudaEvent_t values
 * created and owned by the caller. Pass NULL, NULL to stop recording. Process-wide setting, not
 * synchronised: set it from the thread that issues the calls. Returns FFD_OK, or
 * FFD_ERR_INVALID_ARG when exactly one event is NULL.
 */
ffd_status ffd_set_profile_events(void *start, void *stop);

/*
 * ffd_get_error -- synchronise `stream`, read and clear the device error word at `error_word`
 * (a workspace pointer, or the quantiser's error word), and return FFD_OK, FFD_ERR_BOUNDS or
 * FFD_ERR_RANGE or FFD_ERR_TIMEOUT (in that order of precedence when several bits are set), or
 * FFD_ERR_CUDA if the read failed.
 */
ffd_status ffd_get_error(void *error_word, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FFD_H */
