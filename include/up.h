/*
 * up.h -- C ABI of the UniPrefill block-sparsification hot path for GB300 (sm_103a).
 *
 * UniPrefill drops unimportant tokens during long-context prefill.  At one
 * full-attention layer the last n queries of each sequence score fixed blocks
 * of G key tokens; the highest-scoring blocks are kept until their cumulative
 * score reaches p; the hidden states and position ids of the kept tokens are
 * gathered into a compacted batch that every later layer consumes.
 *
 * Sources: "UniPrefill: 블록 단위 동적 희소화를 통한 범용적 롱 컨텍스트 프리필 가속화"
 * (aitrends.kr overview; paragraphs on block-wise importance estimation, top-p
 * selection, system integration and sparsity propagation) and the UniPrefill
 * abstract (chatpaper.ai; continuous-batching operator).
 *
 * Conventions shared by every call
 *   - All pointers are DEVICE pointers unless stated otherwise.  The caller
 *     allocates and owns every buffer, including the workspace.  The library
 *     never allocates, frees or synchronises; every call is asynchronous and
 *     ordered on `stream`.
 *   - Sequences are continuously batched (varlen): `cu_seqlens` is int32
 *     [num_seqs + 1], cu_seqlens[0] = 0, non-decreasing, and
 *     cu_seqlens[num_seqs] = total_tokens.  L_s = cu_seqlens[s+1] - cu_seqlens[s].
 *   - Tensors are token-major, row-major and contiguous; "bf16" buffers hold
 *     IEEE bfloat16 values.
 *   - nb_s = ceil(L_s / G) blocks per sequence; cu_blocks is int32
 *     [num_seqs + 1], the exclusive prefix sum of nb_s.
 *   - Host-checkable arguments are validated before any launch; a rejected
 *     call launches nothing and returns the error.  Errors found on the device
 *     (a malformed cu_seqlens, a sequence beyond a kernel's size limit, a
 *     page index outside the key pool, an expired bounded wait) set a sticky
 *     device error word that
 *     up_get_device_error() reports; the affected outputs are then unspecified.
 *   - Functions are thread-safe; the first call on a device queries its
 *     attributes and sets kernel attributes for it.
 */
#ifndef UP_H_
#define UP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *up_stream_t;

typedef enum {
    UP_OK = 0,
    UP_ERR_INVALID_ARG = 1,  /* null pointer, bad size, p out of range, misaligned buffer */
    UP_ERR_UNSUPPORTED = 2,  /* valid but outside what the kernels implement (head_dim, G, ...) */
    UP_ERR_WORKSPACE = 3,    /* workspace pointer null or smaller than the *_workspace() size */
    UP_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed (launch, attribute, tensor map) */
    UP_ERR_TIMEOUT = 5,      /* a bounded device-side wait expired (reported by up_get_device_error) */
    UP_ERR_DEVICE = 6        /* a device-side argument check failed (reported by up_get_device_error) */
} up_status;

/* Device error bits reported by up_get_device_error(). */
#define UP_DEVERR_BAD_CU_SEQLENS 0x1u  /* cu_seqlens[0] != 0, decreasing, or last != total_tokens */
#define UP_DEVERR_SELECT_TOO_MANY_BLOCKS 0x2u /* a sequence has more than UP_SELECT_MAX_BLOCKS blocks */
#define UP_DEVERR_TIMEOUT 0x4u         /* a bounded wait inside a kernel gave up */
#define UP_DEVERR_BAD_PAGE 0x8u        /* a page index outside [0, num_pages) (read as zeros) */
#define UP_DEVERR_BAD_CU_BLOCKS 0x10u  /* compaction: cu_blocks[num_seqs] < 0 or > total_tokens/G + num_seqs */
#define UP_DEVERR_BOUNDS 0x20u         /* checked builds only (compiled with -DUP_CHECK_BOUNDS): an index
                                          range outside its buffer; the access was skipped */

/* Largest nb_s that the selection calls rank on chip (1M tokens at G = 64). */
#define UP_SELECT_MAX_BLOCKS 16384

/* Static text for a status code. */
const char *up_status_string(up_status status);

/*
 * Block scoring.
 *
 * Source: UniPrefill overview, block-wise importance estimation paragraph (the
 * last n queries are dotted with all keys; block scores come from softmax
 * attention mass) and drop-criterion paragraph (tokens whose softmax
 * probability is near zero are dropped).
 *
 * For sequence s let n_s = min(n, L_s).  Query t in [0, n_s) sits at absolute
 * position a_t = L_s - n_s + t and sees keys i <= a_t (causal).  For query head
 * h (KV head j = h / (Hq/Hk)):
 *     P[h,t,i] = softmax_i( q[t,h,:] . k[i,j,:] / sqrt(d) )   over i <= a_t
 *     scores[cu_blocks[s] + b] = (1 / (n_s*Hq)) * sum_{h,t} sum_{i in block b} P[h,t,i]
 * so each sequence's scores sum to 1.  Block b covers tokens [bG, min((b+1)G, L_s)).
 *
 *   q_last     bf16 [sum_s n_s, Hq, d]: the last n_s query rows of every
 *              sequence, packed in sequence order (RoPE already applied).
 *   k          bf16 [total_tokens, Hk, d] keys (RoPE already applied).
 *   cu_seqlens int32 [num_seqs+1].
 *   Hq, Hk     query / KV heads, Hq % Hk == 0, Hq/Hk <= 16.
 *   d          head_dim: 64, 128 or 256.
 *   n          observation window (last queries), 1 <= n <= 1024.
 *   G          block size: 16, 32, 64, 128 or 256.
 *   scores     fp32 [sum_s nb_s] (output).  Capacity needed: at most
 *              total_tokens/G + num_seqs entries.
 *   cu_blocks  int32 [num_seqs+1] (output).
 *   workspace  device scratch of at least up_score_blocks_workspace(...) bytes,
 *              256-byte aligned; its contents on entry do not matter.
 * Scores are deterministic: a repeat call on the same inputs returns the same bits.
 */
size_t up_score_blocks_workspace(int num_seqs, int64_t total_tokens, int Hq, int Hk, int d,
                                 int n, int G);

up_status up_score_blocks(const void *q_last, const void *k, const int32_t *cu_seqlens,
                          int num_seqs, int64_t total_tokens, int Hq, int Hk, int d, int n,
                          int G, float *scores, int32_t *cu_blocks, void *workspace,
                          size_t workspace_bytes, up_stream_t stream);

/*
 * Block scores of one tensor-parallel shard of the heads.
 *
 * Source: UniPrefill overview, fused-kernel paragraph: under tensor
 * parallelism each rank scores the heads it holds and the block scores are
 * summed across ranks (an all-reduce) before the selection.
 *
 * Exactly up_score_blocks for the Hq query / Hk KV heads this rank holds
 * (q_last [sum n_s, Hq, d], k [total_tokens, Hk, d], whole GQA groups), except
 * that the mean over heads divides by Hq_total, the query heads of all ranks:
 * score_b = sum over this shard's rows of the block's softmax mass, divided by
 * n_s * Hq_total.  The sum of these scores over a partition of all heads into
 * shards is the up_score_blocks score of all heads (up to fp32 rounding); each
 * shard's scores sum to Hq / Hq_total per sequence.  Hq_total == Hq gives
 * up_score_blocks bit for bit.  Same workspace (up_score_blocks_workspace with
 * this shard's Hq, Hk), outputs and errors as up_score_blocks, plus
 * UP_ERR_INVALID_ARG for Hq_total < Hq.
 */
up_status up_score_blocks_shard(const void *q_last, const void *k, const int32_t *cu_seqlens,
                                int num_seqs, int64_t total_tokens, int Hq, int Hk, int d, int n,
                                int G, int Hq_total, float *scores, int32_t *cu_blocks,
                                void *workspace, size_t workspace_bytes, up_stream_t stream);

/*
 * Block scores with the keys in a paged KV cache (chunked prefill).
 *
 * Sources: Chunked Prefill glossary, how-chunking-works section (a long prompt
 * is prefilled in chunks and each chunk attends to the cached keys of the
 * earlier ones); CompactAttention review, key-terms section (paged attention
 * over a KV-head-major cache).
 *
 * Exactly up_score_blocks, except where the keys are read: key t of sequence s
 * (0 <= t < L_s) is row t % page_size of KV head j in page
 * block_table[s * max_pages + t / page_size] of
 *   k_pages   bf16 [num_pages, Hk, page_size, d]  (KV-head-major pages).
 * The query rows of a chunk are its last n_s tokens, as for up_score_blocks,
 * and a sequence's keys are all of its cached tokens, earlier chunks first.
 *   block_table  int32 [num_seqs * max_pages]; entries past a sequence's pages
 *                are not read.
 *   page_size    a multiple of 128 (a 128-key step never straddles two pages).
 * Errors: as up_score_blocks; UP_ERR_INVALID_ARG for a null table, page_size
 * not a positive multiple of 128, num_pages < 1, num_pages * Hk * page_size
 * >= 2^31, or max_pages < 1; a sequence with more than max_pages * page_size
 * tokens sets UP_DEVERR_BAD_CU_SEQLENS (nothing is scored); a page index
 * outside [0, num_pages) sets UP_DEVERR_BAD_PAGE and its keys read as zeros.
 * The workspace is up_score_blocks_workspace's.
 */
up_status up_score_blocks_paged(const void *q_last, const void *k_pages, int64_t num_pages,
                                int page_size, const int32_t *block_table, int max_pages,
                                const int32_t *cu_seqlens, int num_seqs, int64_t total_tokens,
                                int Hq, int Hk, int d, int n, int G, float *scores,
                                int32_t *cu_blocks, void *workspace, size_t workspace_bytes,
                                up_stream_t stream);

/*
 * The kept blocks as a block-CSR matrix (sequences x key blocks) for a
 * block-sparse attention consumer.
 *
 * Source: FlashPrefill V2 review, key-terms section (the active blocks are
 * handed to the sparse-attention kernel as a CSR index).
 *
 *   keep, cu_blocks  as produced by up_select_topp / up_select_blocks and
 *                    up_score_blocks (cu_blocks int32 [num_seqs+1]).
 *   indptr   int32 [num_seqs+1] (output): indptr[s] = kept blocks of the
 *            sequences before s; indptr[num_seqs] = all kept blocks.
 *   indices  int32 [sum nb_s] (output, capacity): entries indptr[s] ..
 *            indptr[s+1]-1 are the kept block numbers of sequence s (0-based
 *            within the sequence), ascending.
 * One CTA; no workspace.  Errors: UP_ERR_INVALID_ARG for a null pointer or
 * num_seqs < 0.
 */
up_status up_block_csr(const uint8_t *keep, const int32_t *cu_blocks, int num_seqs,
                       int32_t *indptr, int32_t *indices, up_stream_t stream);

/*
 * Top-p block selection.
 *
 * Source: UniPrefill overview, top-p selection paragraph: blocks sorted by
 * score are kept until their cumulative sum reaches p (e.g. 0.99).
 *
 * Per sequence, blocks are ranked by (score descending, block index
 * ascending); the cumulative score is taken exactly in rank order (each fp32
 * score as a 64-bit fixed-point multiple of 2^-62, truncated); the kept set is
 * the shortest prefix whose cumulative score is >= p, crossing block included
 * (block at rank r kept iff the mass ranked before it is < ceil(p * 2^62)).
 * p >= 1 keeps every block; if rounding leaves the total below p, every block
 * is kept.
 *
 *   scores, cu_blocks  as produced by up_score_blocks: block masses >= 0 that
 *                      sum to about 1 per sequence (a score >= 1 counts as 1;
 *                      a total above 2 gives an unspecified kept set).
 *   cu_seqlens         int32 [num_seqs+1] (block lengths for kept_tokens).
 *   p                  0 < p; p >= 1 keeps all.
 *   keep               uint8 [sum nb_s] (output): 1 kept, 0 dropped, original order.
 *   kept_tokens        int32 [num_seqs] (output): tokens in the kept blocks.
 * Sequences with nb_s > UP_SELECT_MAX_BLOCKS raise UP_DEVERR_SELECT_TOO_MANY_BLOCKS.
 */
up_status up_select_topp(const float *scores, const int32_t *cu_blocks,
                         const int32_t *cu_seqlens, int num_seqs, int G, double p,
                         uint8_t *keep, int32_t *kept_tokens, up_stream_t stream);

/* Selection rule of up_select_blocks. */
typedef enum { UP_SELECT_TOP_P = 0, UP_SELECT_TOP_K = 1 } up_select_mode;

/* up_select_blocks flag: also keep the last block of every non-empty sequence. */
#define UP_SELECT_KEEP_LAST 0x1u

/*
 * Block selection, general form.
 *
 * Sources: UniPrefill overview, top-p selection paragraph (top-p),
 * hyper-parameters paragraph (its ablation sets top-p against keeping a fixed
 * number of blocks: top-k), system-integration paragraph (decode continues
 * from the end of each sequence: the keep-last option).
 *
 * Blocks are ranked per sequence exactly as in up_select_topp (score
 * descending, block index ascending).
 *   mode UP_SELECT_TOP_P  the kept set of up_select_topp with threshold p
 *                         (0 < p; k is ignored).
 *   mode UP_SELECT_TOP_K  the first min(k, nb_s) ranks (k >= 1; p is ignored).
 *   flags                 0, or UP_SELECT_KEEP_LAST: after the rule, the last
 *                         block of every non-empty sequence is kept too and
 *                         counted in kept_tokens (the method as the pages state
 *                         it leaves this off).
 * The other arguments, outputs and device errors are those of up_select_topp;
 * an unknown mode or flag bit, p <= 0 or NaN in top-p mode, or k < 1 in top-k
 * mode return UP_ERR_INVALID_ARG before any launch.
 */
up_status up_select_blocks(const float *scores, const int32_t *cu_blocks,
                           const int32_t *cu_seqlens, int num_seqs, int G, up_select_mode mode,
                           double p, int k, uint32_t flags, uint8_t *keep, int32_t *kept_tokens,
                           up_stream_t stream);

/*
 * Compaction (sparsity propagation).
 *
 * Source: UniPrefill overview, sparsity-propagation paragraph (every later
 * sub-layer takes only the kept tokens) and system-integration paragraph (the
 * positions of dropped/kept tokens travel with the batch so decode addresses
 * the right KV-cache slots).
 *
 * For each sequence in order and each kept block in ascending order, the
 * block's rows of x and pos are appended to x_out / pos_out.  Positions are
 * gathered, not renumbered.
 *
 *   x               bf16 [total_tokens, hidden], 16-byte aligned; hidden % 8 == 0.
 *   pos             int32 [total_tokens].
 *                   x and pos may be device memory, or pinned (page-locked) host
 *                   memory that the device addresses through unified addressing
 *                   (cudaHostAlloc, cudaHostRegister): the kernel then reads only
 *                   the kept rows across the host link, in place.
 *   keep, cu_blocks as produced above.
 *   x_out           bf16 [capacity, hidden], 16-byte aligned; capacity must be
 *                   >= the number of kept tokens (total_tokens is always enough).
 *   pos_out         int32 [capacity].
 *   cu_seqlens_out  int32 [num_seqs+1] (output): cu_seqlens of the compacted batch.
 *   src_idx         int32 [capacity] or NULL: source row of every output row.
 *   total_kept      int32 [1] (output): number of kept rows (= cu_seqlens_out[num_seqs]).
 *   workspace       at least up_compact_workspace(...) bytes, 256-byte aligned.
 * The output size lives on the device; reading it on the host is the caller's
 * choice (one device-to-host copy of total_kept).  A cu_blocks that cannot be
 * this batch's (its last entry negative or above total_tokens/G + num_seqs;
 * for one sequence, anything but {0, ceil(total_tokens/G)}) sets
 * UP_DEVERR_BAD_CU_BLOCKS and total_kept is 0; nothing is read or written out
 * of bounds, and the other outputs are unspecified.
 */
size_t up_compact_workspace(int num_seqs, int64_t total_tokens, int G);

up_status up_compact(const void *x, const int32_t *pos, int hidden, const int32_t *cu_seqlens,
                     int num_seqs, int64_t total_tokens, int G, const uint8_t *keep,
                     const int32_t *cu_blocks, void *x_out, int32_t *pos_out,
                     int32_t *cu_seqlens_out, int32_t *src_idx, int32_t *total_kept,
                     void *workspace, size_t workspace_bytes, up_stream_t stream);

/*
 * Compaction without a caller-supplied workspace.
 *
 * The UniPrefill pages have no counterpart of this entry point; it exists for
 * callers that cannot allocate device memory when they compact -- an engine
 * that has reserved nearly all HBM for its KV cache, or a serving loop that
 * must not call cudaMalloc because it can synchronise the device.
 *
 * It computes exactly what up_compact computes, with the same arguments minus
 * the workspace.  Its scratch (kept-block list, per-block destination rows and
 * a counter, about 1.3 MB) is a fixed array inside the library that every GPU
 * loading the library holds until the process exits; the call itself
 * allocates and frees nothing.
 *   - Limit: total_tokens / G + num_seqs <= UP_COMPACT_NOALLOC_MAX_BLOCKS
 *     (4M tokens at G = 64); larger batches return UP_ERR_WORKSPACE and launch
 *     nothing.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - All calls on a device share the one array.  Each call rewrites every
 *     scratch entry it reads, so no clearing is needed, but calls that overlap
 *     on the GPU (different streams, no ordering between them) race on it and
 *     give wrong results.
 */
#define UP_COMPACT_NOALLOC_MAX_BLOCKS 65536

up_status up_compact_noalloc(const void *x, const int32_t *pos, int hidden,
                             const int32_t *cu_seqlens, int num_seqs, int64_t total_tokens, int G,
                             const uint8_t *keep, const int32_t *cu_blocks, void *x_out,
                             int32_t *pos_out, int32_t *cu_seqlens_out, int32_t *src_idx,
                             int32_t *total_kept, up_stream_t stream);

/*
 * Instrumentation: when both events are non-NULL, every later scoring call
 * (up_score_blocks, up_score_blocks_shard, up_score_blocks_paged) made by this
 * host thread records `start_event` immediately before its
 * tensor-core scoring kernel and `stop_event` immediately after it, on the
 * call's stream, so the caller can time that kernel alone with
 * cudaEventElapsedTime.  Pass NULL, NULL to stop.  The events are cudaEvent_t
 * handles owned by the caller.  Not part of the method; no page counterpart.
 */
typedef struct CUevent_st *up_event_t;
up_status up_set_kernel_timing_events(up_event_t start_event, up_event_t stop_event);

/*
 * Instrumentation: measures this GPU's sustained MUFU ex2 rate (exponentials
 * per second over the whole device) with a short full-occupancy kernel on
 * `stream`, and writes it to *ex2_per_second.  Synchronises the stream (about
 * a millisecond).  This is the exponential roof of up_score_blocks, which
 * evaluates one ex2 per visible (query head, query, key) triple.  Not part of
 * the method; no page counterpart.
 */
up_status up_measure_ex2_rate(double *ex2_per_second, up_stream_t stream);

/*
 * Instrumentation for tests of the failure path: every spin-wait inside the
 * tensor-core scoring kernel (a role waiting for shared-memory data, a free
 * TMEM buffer or another CTA's results) gives up after `cycles` SM clock
 * cycles; the kernel then stops every role of the CTA, lets its copies and
 * MMAs in flight complete, frees its tensor memory, returns and sets
 * UP_DEVERR_TIMEOUT (the call's outputs are then unspecified).  0 restores
 * the default bound (4e9 cycles, about two seconds); a bound above the
 * default returns UP_ERR_INVALID_ARG.  Process-wide; it applies to scoring
 * calls issued after it.  Not part of the method; no page counterpart.
 */
up_status up_set_wait_limit(uint64_t cycles);

/*
 * Reads and clears the sticky device error word of the current device
 * (UP_DEVERR_* bits; 0 if none).  This call synchronises the device.
 * Returns UP_OK if no bit was set, UP_ERR_TIMEOUT if the timeout bit was set,
 * UP_ERR_DEVICE for any other bit, UP_ERR_CUDA if the copy itself failed.
 */
up_status up_get_device_error(uint32_t *bits);

#ifdef __cplusplus
}
#endif

#endif /* UP_H_ */
