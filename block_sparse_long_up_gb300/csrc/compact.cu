// compact.cu -- gather the kept tokens' hidden states and positions.
//
// UniPrefill overview, sparsity-propagation paragraph: every later sub-layer
// takes only the kept tokens; system-integration paragraph: the kept tokens'
// positions travel with them.  A kept block is a contiguous run of at most G
// rows, so compaction is a set of contiguous copies.
//
// One kernel (batches of at most kCompactOneKernelBlocks blocks): every CTA
// scans the keep flags itself -- thread t counts the kept rows of a contiguous
// range of blocks and one CTA-wide scan gives each range its first output row
// and the total T -- and then copies the output rows [c*T/F, (c+1)*T/F) of its
// own share (F CTAs), so the work is split by bytes, not by blocks.  The scan
// is repeated by every CTA (a few KB of flags from L2) instead of being handed
// from one kernel to the next through memory: that saves a launch and a chain
// of dependent global loads.  CTA 0 also writes cu_seqlens_out and the total.
//
// Two kernels (larger batches): an index kernel (one CTA, the same scan) writes
// the kept-block list (source row, destination row, rows) to scratch memory,
// and a persistent gather copies it in work items of a few rows.
//
// Also here: the kept blocks as a block-CSR matrix for a sparse-attention
// consumer (FlashPrefill V2 review, key-terms section), by the same scan.
#include "../../include/up.h"
#include "common.cuh"

namespace up {

namespace {

constexpr int kIndexThreads = 1024;
constexpr int kGatherThreads = 512;
constexpr int kOneThreads = 512;
constexpr int kOnePieces = 2048;  // copy pieces one CTA can hold (its rows, at most)

// Block-wide exclusive scan of one int64 per thread (blockDim.x a multiple of
// 32, at most 1024).  sh holds 32 entries.
__device__ int64_t block_excl_scan_i64(int64_t v, int64_t *total, int64_t *sh) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int nw = (int)(blockDim.x >> 5);
    int64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int64_t w = lane < nw ? sh[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        sh[lane] = w;
    }
    __syncthreads();
    *total = sh[nw - 1];
    return (wid ? sh[wid - 1] : 0) + x - v;
}

// The sequence holding global block gb (the last one starting at or before it).
__device__ __forceinline__ int seq_of_block(const int32_t *cu_blocks, int B, int gb) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu_blocks[mid] <= gb) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Rows of block gb of sequence s.
__device__ __forceinline__ int block_rows(const CompactArgs &a, int s, int gb) {
    return min(a.G, a.cu_seqlens[s + 1] - a.cu_seqlens[s] - (gb - a.cu_blocks[s]) * a.G);
}

// cu_blocks[B] must be a block count the batch can have; anything else would
// send the scan (and the two-kernel path's scratch writes) out of bounds.
__device__ __forceinline__ bool block_count_ok(const CompactArgs &a, int nbt) {
    return nbt >= 0 && (int64_t)nbt <= a.max_blocks;
}

// 16-byte copy of nv vectors by all NT threads of the CTA, eight loads in
// flight per thread (at a few rows per CTA the whole copy is one round trip).
// NT is a constant, so the eight addresses are one base plus immediate offsets.
template <int NT>
__device__ __forceinline__ void copy_vec(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                         int64_t nv) {
    constexpr int kU = 8;
    for (int64_t v0 = 0; v0 < nv; v0 += kU * NT) {
        const uint4 *s = src + v0 + threadIdx.x;
        uint4 *d = dst + v0 + threadIdx.x;
        const int64_t left = nv - v0 - threadIdx.x;  // vectors from this thread's first one
        uint4 x[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u)
            if (u * NT < left) x[u] = __ldcs(s + u * NT);
#pragma unroll
        for (int u = 0; u < kU; ++u)
            if (u * NT < left) __stcs(d + u * NT, x[u]);
    }
}

__global__ void __launch_bounds__(kOneThreads, 2)
compact_one_kernel(CompactArgs a) {
    __shared__ int64_t scan_sh[32];
    __shared__ int rstart[kOneThreads];     // first output row of each thread's block range
    __shared__ int4 piece[kOnePieces];      // (source row, output row, rows, -)
    __shared__ int npiece;
    pdl_wait();
    const int B = a.num_seqs, t = threadIdx.x;
    // one sequence: the block count is the host's (the flags' loads need not
    // wait for cu_blocks); cu_blocks[1] is still checked against it, below
    const bool one = a.nb_one >= 0;
    const int nbt = one ? a.nb_one : a.cu_blocks[B];
    if (!block_count_ok(a, nbt)) {
        if (blockIdx.x == 0 && t == 0) {
            atomicOr(a.err, UP_DEVERR_BAD_CU_BLOCKS);
            *a.total_kept = 0;
        }
        return;
    }
    const int L0 = one ? a.cu_seqlens[1] - a.cu_seqlens[0] : 0;
    const int per = (nbt + kOneThreads - 1) / kOneThreads;
    const int g0 = min(t * per, nbt), g1 = min(g0 + per, nbt);
    const int s0 = g0 < g1 && !one ? seq_of_block(a.cu_blocks, B, g0) : 0;
    auto rows_of = [&](int s, int gb) { return one ? min(a.G, L0 - gb * a.G) : block_rows(a, s, gb); };
    int rows = 0;
    for (int gb = g0, s = s0; gb < g1; ++gb) {
        if (!one)
            while (a.cu_blocks[s + 1] <= gb) ++s;
        if (a.keep[gb]) rows += rows_of(s, gb);
    }
    int64_t T64;
    const int first = (int)block_excl_scan_i64(rows, &T64, scan_sh);
    const int T = (int)T64;
    rstart[t] = first;
    if (t == 0) npiece = 0;
    __syncthreads();
    // this CTA's output rows
    const int lo = (int)((int64_t)T * blockIdx.x / gridDim.x);
    const int hi = (int)((int64_t)T * (blockIdx.x + 1) / gridDim.x);
    if (first < hi && first + rows > lo) {
        int dst = first;
        for (int gb = g0, s = s0; gb < g1 && dst < hi; ++gb) {
            if (!one)
                while (a.cu_blocks[s + 1] <= gb) ++s;
            if (!a.keep[gb]) continue;
            const int len = rows_of(s, gb);
            if (dst + len > lo) {
                const int c0 = max(dst, lo), c1 = min(dst + len, hi);
                const int src = (one ? a.cu_seqlens[0] + gb * a.G
                                     : a.cu_seqlens[s] + (gb - a.cu_blocks[s]) * a.G) +
                                (c0 - dst);
                const int i = atomicAdd(&npiece, 1);
                if (i < kOnePieces) piece[i] = make_int4(src, c0, c1 - c0, 0);
            }
            dst += len;
        }
    }
    __syncthreads();
    const int np = min(npiece, kOnePieces);  // <= hi - lo <= kOnePieces by the grid size
    for (int i = 0; i < np; ++i) {
        const int4 e = piece[i];
        if (!in_range(e.x, e.z, a.total_tokens, a.err) || !in_range(e.y, e.z, a.total_tokens, a.err))
            continue;
        copy_vec<kOneThreads>(a.x + (int64_t)e.x * a.vec_per_row,
                              a.x_out + (int64_t)e.y * a.vec_per_row, (int64_t)e.z * a.vec_per_row);
        for (int r = t; r < e.z; r += kOneThreads) {
            a.pos_out[e.y + r] = a.pos[e.x + r];
            if (a.src_idx) a.src_idx[e.y + r] = e.x + r;
        }
    }
    if (blockIdx.x == 0) {
        // one sequence: cu_blocks must be {0, nbt} (the batch's own)
        const bool bad = one && (a.cu_blocks[0] != 0 || a.cu_blocks[1] != nbt);
        if (bad && t == 0) atomicOr(a.err, UP_DEVERR_BAD_CU_BLOCKS);
        // cu_seqlens_out[s]: the output row of sequence s's first block -- the
        // first row of the range holding it plus the kept rows before it there
        for (int s = t; s <= B; s += kOneThreads) {
            const int b = max(a.cu_blocks[s], 0);
            int v = T;
            if (b < nbt) {
                const int u = b / per;
                v = rstart[u];
                for (int gb = u * per; gb < b; ++gb)
                    if (a.keep[gb]) v += block_rows(a, seq_of_block(a.cu_blocks, B, gb), gb);
            }
            a.cu_out[s] = v;
        }
        if (t == 0) *a.total_kept = bad ? 0 : T;
    }
}

// Thread t takes a contiguous range of blocks: it counts the kept rows and
// blocks of its range, one block-wide scan of the (rows, blocks) pair gives its
// starting destination row and list slot, and it writes its range.
__global__ void __launch_bounds__(kIndexThreads)
compact_index_kernel(CompactArgs a) {
    pdl_wait();
    __shared__ int64_t sh[32];
    const int B = a.num_seqs;
    const int nbt = a.cu_blocks[B];
    if (!block_count_ok(a, nbt)) {
        if (threadIdx.x == 0) {
            atomicOr(a.err, UP_DEVERR_BAD_CU_BLOCKS);
            *a.total_kept = 0;
            *a.nkept = 0;  // the gather copies nothing
        }
        return;
    }
    const int per = (nbt + kIndexThreads - 1) / kIndexThreads;
    const int g0 = min((int)threadIdx.x * per, nbt), g1 = min(g0 + per, nbt);
    const int s0 = g0 < g1 ? seq_of_block(a.cu_blocks, B, g0) : 0;
    int rows = 0, kb = 0;
    for (int gb = g0, s = s0; gb < g1; ++gb) {
        while (a.cu_blocks[s + 1] <= gb) ++s;
        if (a.keep[gb]) {
            rows += block_rows(a, s, gb);
            ++kb;
        }
    }
    // rows in the high word, kept blocks in the low word (neither sum can carry)
    int64_t tot;
    const int64_t ex = block_excl_scan_i64(((int64_t)rows << 32) | kb, &tot, sh);
    int dst = (int)(ex >> 32), slot = (int)(ex & 0xFFFFFFFF);
    for (int gb = g0, s = s0; gb < g1; ++gb) {
        while (a.cu_blocks[s + 1] <= gb) ++s;
        a.dst_blk[gb] = dst;
        if (a.keep[gb]) {
            const int len = block_rows(a, s, gb);
            a.list[slot++] = make_int4(a.cu_seqlens[s] + (gb - a.cu_blocks[s]) * a.G, dst, len, 0);
            dst += len;
        }
    }
    const int total_rows = (int)(tot >> 32);
    __syncthreads();
    for (int s = threadIdx.x; s <= B; s += kIndexThreads) {
        const int cb = a.cu_blocks[s];
        a.cu_out[s] = cb < nbt ? a.dst_blk[cb] : total_rows;
    }
    if (threadIdx.x == 0) {
        *a.total_kept = total_rows;
        *a.nkept = (int)(tot & 0xFFFFFFFF);
    }
}

__global__ void __launch_bounds__(kGatherThreads)
compact_gather_kernel(CompactArgs a) {
    pdl_wait();
    const int K = *a.nkept;
    if (!in_range(0, K, a.max_blocks, a.err)) return;  // checked builds: the list's length
    const int64_t items = (int64_t)K * a.items_per_block;
    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        const int kb = (int)(it / a.items_per_block);
        const int q = (int)(it % a.items_per_block);
        const int4 e = a.list[kb];  // src row, dst row, rows
        const int r0 = q * a.rows_per_item;
        if (r0 >= e.z) continue;
        const int rows = min(e.z - r0, a.rows_per_item);
        if (!in_range(e.x + r0, rows, a.total_tokens, a.err) ||
            !in_range(e.y + r0, rows, a.total_tokens, a.err))
            continue;
        copy_vec<kGatherThreads>(a.x + (int64_t)(e.x + r0) * a.vec_per_row,
                                 a.x_out + (int64_t)(e.y + r0) * a.vec_per_row,
                                 (int64_t)rows * a.vec_per_row);
        if (threadIdx.x < rows) {
            const int sr = e.x + r0 + threadIdx.x, dr = e.y + r0 + threadIdx.x;
            a.pos_out[dr] = a.pos[sr];
            if (a.src_idx) a.src_idx[dr] = sr;
        }
    }
}

// Block CSR of the kept blocks (one CTA): thread t takes a contiguous run of
// blocks and counts its kept ones, one block-wide scan gives each run's first
// output slot (kept in shared memory), and each thread writes its kept block
// numbers.  indptr[s] is the slot of the sequence's first block: the run that
// holds it plus the kept blocks of that run before it.
__global__ void __launch_bounds__(kIndexThreads)
block_csr_kernel(const uint8_t *__restrict__ keep, const int32_t *__restrict__ cu_blocks,
                 int B, int32_t *__restrict__ indptr, int32_t *__restrict__ indices) {
    pdl_wait();
    __shared__ int64_t sh[32];
    __shared__ int start[kIndexThreads];
    const int nbt = cu_blocks[B];
    const int per = (nbt + kIndexThreads - 1) / kIndexThreads;
    const int g0 = min((int)threadIdx.x * per, nbt), g1 = min(g0 + per, nbt);
    int cnt = 0;
    for (int gb = g0; gb < g1; ++gb) cnt += keep[gb] != 0;
    int64_t tot;
    const int first = (int)block_excl_scan_i64(cnt, &tot, sh);
    start[threadIdx.x] = first;
    if (g0 < g1) {
        int pos = first;
        for (int gb = g0, s = seq_of_block(cu_blocks, B, g0); gb < g1; ++gb) {
            while (cu_blocks[s + 1] <= gb) ++s;
            if (keep[gb]) indices[pos++] = gb - cu_blocks[s];
        }
    }
    __syncthreads();
    for (int s = threadIdx.x; s <= B; s += kIndexThreads) {
        const int b = cu_blocks[s];
        int v = (int)tot;
        if (b < nbt) {
            const int u = b / per;  // the run holding block b
            v = start[u];
            for (int gb = u * per; gb < b; ++gb) v += keep[gb] != 0;
        }
        indptr[s] = v;
    }
}

}  // namespace

cudaError_t launch_compact(const CompactArgs &a, int num_sms, cudaStream_t st) {
    if (a.max_blocks <= kCompactOneKernelBlocks) {
        // two CTAs per SM; more CTAs only when one CTA's share of the rows
        // could exceed its piece table (every kept row is a piece at worst)
        const int64_t rows_max = a.max_blocks * a.G;
        int64_t grid = 2 * (int64_t)num_sms;
        const int64_t need = (rows_max + kOnePieces - 1) / kOnePieces;
        if (grid < need) grid = need;
        if (grid < 1) grid = 1;
        return launch_pdl(compact_one_kernel, dim3((unsigned)grid), dim3(kOneThreads), 0, st, a);
    }
    cudaError_t e = launch_pdl(compact_index_kernel, dim3(1), dim3(kIndexThreads), 0, st, a);
    if (e != cudaSuccess) return e;
    return launch_pdl(compact_gather_kernel, dim3(num_sms * 4), dim3(kGatherThreads), 0, st, a);
}

cudaError_t launch_block_csr(const uint8_t *keep, const int32_t *cu_blocks, int num_seqs,
                             int32_t *indptr, int32_t *indices, cudaStream_t st) {
    return launch_pdl(block_csr_kernel, dim3(1), dim3(kIndexThreads), 0, st, keep, cu_blocks,
                      num_seqs, indptr, indices);
}

}  // namespace up
