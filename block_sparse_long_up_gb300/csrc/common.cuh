// common.cuh -- internal types shared by the kernels of the UniPrefill hot path.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace up {

// Programmatic dependent launch.  Every kernel of the library is launched with
// the attribute and calls pdl_wait() before it reads what the previous kernel
// of the stream wrote: that waits until that kernel has finished and its
// writes are visible (read-after-write and write-after-read alike).  A kernel
// that calls pdl_trigger() lets the next kernel's CTAs be scheduled while it
// still runs; one that does not releases them as its CTAs exit.  Only the
// one-warp plan kernel triggers early, right after its own pdl_wait(): every
// kernel before it is then complete, so the scoring kernel may read the call's
// inputs (q_last, k, cu_seqlens) and write its own workspace regions before it
// waits for the plan itself.  Everywhere else early-scheduled CTAs that only
// wait measured slower than a release at exit.  Both calls are no-ops for a
// kernel launched without the attribute.
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch with programmatic stream serialization (see pdl_wait).
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Per-sequence work description, written on the device by the plan kernel from
// cu_seqlens, so the host never needs the sequence lengths.
struct SeqInfo {
    int32_t tok_off;   // cu_seqlens[s]
    int32_t L;         // tokens in the sequence
    int32_t ns;        // min(n, L): scored queries
    int32_t q_off;     // first row of q_last for this sequence
    int32_t nb;        // ceil(L / G)
    int32_t blk_off;   // cu_blocks[s]
    int32_t nchunks;   // ceil(L / C): key chunks
    int32_t mtiles;    // ceil(ceil(ns / tokens_per_tile) / tiles_per_unit): row-tile groups per KV head
    int32_t R;         // Hq * ns: softmax rows of the sequence
    int32_t unit_off;  // first score work unit of the sequence
    int64_t row_off;   // first global row (exclusive prefix of R)
    int64_t part_off;  // first float of the (block, row) partial sums
    int64_t stat_off;  // first float of the (chunk, row) statistics
};
static_assert(sizeof(SeqInfo) == 64, "SeqInfo is 64 bytes");

// Device counters at the head of the score workspace.
struct Counters {
    int32_t units;       // score work units
    int32_t blocks;      // sum nb_s
    int64_t rows;        // sum R_s
    int32_t flagged;     // row tiles queued for the exact fallback
    int32_t bar[3];      // the scoring kernel's grid barriers (CTAs arrived)
    int32_t pad[8];
};
static_assert(sizeof(Counters) == 64, "Counters is 64 bytes");

// Checked builds (-DUP_CHECK_BOUNDS): every kernel tests the index ranges it
// writes or reads against its buffers' sizes, sets UP_DEVERR_BOUNDS and skips
// the access when one falls outside (no trap: the context stays usable).  In
// the normal build the test is a constant true and compiles away.
#ifdef UP_CHECK_BOUNDS
constexpr bool kCheckBounds = true;
#else
constexpr bool kCheckBounds = false;
#endif

// [start, start + len) inside [0, n)?
__device__ __forceinline__ bool in_range(int64_t start, int64_t len, int64_t n,
                                         unsigned int *err) {
    if constexpr (!kCheckBounds) {
        return true;
    } else {
        const bool ok = start >= 0 && len >= 0 && start + len <= n;
        if (!ok) atomicOr(err, 0x20u);  // UP_DEVERR_BOUNDS
        return ok;
    }
}

constexpr int kRowsPerTile = 128;   // rows of one M tile (TMEM lanes)
constexpr int kStepKeys = 128;      // keys of one MMA step (N)

// Softmax rows of a sequence are numbered r = j * g * n_s + t * g + h for query
// t (0..n_s-1) of query head j * g + h (h < g, the GQA group of KV head j):
// token-major inside a group, so one row tile holds the g heads of
// tokens_per_tile consecutive queries (the g heads of a query are adjacent in
// q_last, and a tile is one tensor-map box per 64 head dims).  At most
// 128 - g * tokens_per_tile rows of a tile stay unused when g is not a power of 2.
__host__ __device__ constexpr int tokens_per_tile(int g) { return kRowsPerTile / g; }

// Row tiles a score CTA computes against each key step: all four tiles of a
// 512-row GQA group share every K step in shared memory (head_dim <= 128); at
// head_dim 256 the Q tiles of four would not fit next to the K ring, so two.
__host__ __device__ constexpr int tiles_per_unit(int d) { return d <= 128 ? 4 : 2; }
constexpr int kChunkQuantum = 256;  // key chunks are multiples of this (and of G)
constexpr int kSlotsPerChunk = 1;   // statistics slots per (row, key chunk)

// Statistics slot of block b (C is a multiple of G).
__host__ __device__ __forceinline__ int block_slot(int b, int G, int C) {
    return kSlotsPerChunk * ((b * G) / C);
}

// Score workspace layout (offsets in bytes, every region 256-byte aligned).
struct ScoreLayout {
    size_t seqs, counters, part, mref, lsum, flags, total;
    int64_t max_part, max_stat, max_rows, max_units, max_blocks, total_tokens;
    int64_t max_qrows;  // upper bound on the rows of q_last (sum of n_s)
    int chunk;  // C: keys per work unit
};

// Everything the scoring kernels read.
struct ScoreParams {
    const __nv_bfloat16 *q;
    const __nv_bfloat16 *k;
    const SeqInfo *seqs;
    const Counters *counters;
    const int32_t *cu_seqlens;
    // One sequence: its table row and unit count as the plan computes them from
    // total_tokens (cu_seqlens must then be {0, total_tokens}); unused otherwise.
    SeqInfo seq0;
    int units0;
    float *part;   // [b][r] per sequence: block partial sums (relative to mref)
    float *mref;   // [c][r] per sequence: reference (log2 units) of the chunk's partials,
                   // then (overwritten in place) the weight of the chunk's partials
    float *lsum;   // [c][r] per sequence: sum of the chunk's partials
    float *scores;
    int32_t *flag_list;  // 4*unit + row tile of tiles whose sums overflowed (exact fallback)
    int max_units;
    int flag_cap;        // capacity of flag_list
    int num_seqs, Hq, Hk, g, d, n, G, C;
    int Hq_norm;       // heads the mean over heads divides by (Hq, or all ranks' heads)
    // Paged keys (null block_table: k is token-major [total, Hk, d]).  Key t of
    // sequence s is row t % page_size of head j in page block_table[s*max_pages +
    // t/page_size] of k viewed as [num_pages][Hk][page_size][d].
    const int32_t *block_table;
    int page_size, max_pages;
    int64_t num_pages;
    int tpt;           // tokens_per_tile(g)
    float scale_log2;  // log2(e) / sqrt(d)
    long long wait_limit;  // bound of every spin-wait of the scoring kernel, SM clock cycles
    unsigned int *err;
    int64_t part_cap, stat_cap, scores_cap;  // floats in part, in mref/lsum each, in scores
};

__device__ __forceinline__ int find_seq_by_unit(const SeqInfo *seqs, int B, int u) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (seqs[mid].unit_off <= u) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Row of key `tok` of sequence s, KV head j, in the paged keys viewed as a 2-D
// [num_pages * Hk * page_size, d] array; a page index outside [0, num_pages)
// sets UP_DEVERR_BAD_PAGE and returns the row count (one past the last row).
__device__ __forceinline__ int64_t paged_row(const ScoreParams &p, int s, int j, int tok) {
    const int64_t pg = p.block_table[(int64_t)s * p.max_pages + tok / p.page_size];
    if (pg < 0 || pg >= p.num_pages) {
        atomicOr(p.err, 0x8u);  // UP_DEVERR_BAD_PAGE
        return p.num_pages * p.Hk * p.page_size;
    }
    return (pg * p.Hk + j) * p.page_size + tok % p.page_size;
}

// Host-side launchers (each returns the launch's cudaError_t).
cudaError_t launch_score_plan(const int32_t *cu_seqlens, int32_t *cu_blocks, const ScoreParams &p,
                              int64_t total_tokens, cudaStream_t st);
cudaError_t launch_score_main(const ScoreParams &p, const ScoreLayout &lay, int num_sms,
                              cudaStream_t st);
// top_k: keep the first k ranks (p unused); otherwise top-p with p.
cudaError_t launch_select(const float *scores, const int32_t *cu_blocks, const int32_t *cu_seqlens,
                          int num_seqs, int G, bool top_k, double p, int k, bool keep_last,
                          uint8_t *keep, int32_t *kept_tokens, unsigned int *err, int num_sms,
                          cudaStream_t st);

struct CompactArgs {
    const uint4 *x;
    const int32_t *pos;
    const int32_t *cu_seqlens;
    const uint8_t *keep;
    const int32_t *cu_blocks;
    uint4 *x_out;
    int32_t *pos_out;
    int32_t *cu_out;
    int32_t *src_idx;
    int32_t *total_kept;
    int4 *list;        // scratch (blocks beyond the one-kernel limit): kept blocks (src row, dst row, rows, -)
    int32_t *nkept;    // scratch: number of kept blocks
    int32_t *dst_blk;  // scratch: destination row of every block
    unsigned int *err; // the device error word
    int64_t max_blocks;  // total_tokens / G + num_seqs: the most blocks the batch can have
    int nb_one;          // one sequence: ceil(total_tokens / G), its block count; else -1
    int num_seqs, G, hidden, rows_per_item, items_per_block;
    int64_t vec_per_row;  // hidden * 2 / 16
    int64_t total_tokens; // rows of x and pos (and the most rows x_out can need)
};
// Compaction kernels: one kernel when max_blocks <= kCompactOneKernelBlocks
// (every CTA scans the keep flags itself; the scratch is not used), else an
// index kernel that writes the kept-block list to the scratch and a gather.
constexpr int64_t kCompactOneKernelBlocks = 16384;
cudaError_t launch_compact(const CompactArgs &a, int num_sms, cudaStream_t st);
// The device error word of the current device (nullptr if it cannot be looked up).
unsigned int *device_error_word();
cudaError_t launch_block_csr(const uint8_t *keep, const int32_t *cu_blocks, int num_seqs,
                             int32_t *indptr, int32_t *indices, cudaStream_t st);

}  // namespace up
