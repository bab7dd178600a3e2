// compact.cu -- gather the kept tokens' hidden states and positions.
//
// UniPrefill overview, sparsity-propagation paragraph: every later sub-layer
// takes only the kept tokens; system-integration paragraph: the kept tokens'
// positions travel with them.  A kept block is a contiguous run of at most G
// rows, so compaction is a set of contiguous copies:
//   index  (1 CTA)  one exclusive scan over per-thread block ranges -> kept-block list
//                   (source row, destination row, rows), cu_seqlens_out, total;
//   gather (persistent grid) one work item = up to rows_per_item rows of one
//                   kept block, copied with 16-byte vector loads and stores.
// Also here: the kept blocks as a block-CSR matrix for a sparse-attention
// consumer (FlashPrefill V2 review, key-terms section), by the same scan.
#include "common.cuh"

namespace up {

namespace {

constexpr int kIndexThreads = 1024;
constexpr int kGatherThreads = 512;

// Block-wide exclusive scan of one int64 per thread (blockDim.x == 1024).
__device__ int64_t block_excl_scan_i64(int64_t v, int64_t *total, int64_t *sh) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int64_t w = sh[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        sh[lane] = w;
    }
    __syncthreads();
    *total = sh[31];
    return (wid ? sh[wid - 1] : 0) + x - v;
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
    const int per = (nbt + kIndexThreads - 1) / kIndexThreads;
    const int g0 = min((int)threadIdx.x * per, nbt), g1 = min(g0 + per, nbt);
    int s0 = 0;  // the sequence holding block g0 (the last one starting at or before it)
    if (g0 < g1) {
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (a.cu_blocks[mid] <= g0) lo = mid; else hi = mid - 1;
        }
        s0 = lo;
    }
    int rows = 0, kb = 0;
    for (int gb = g0, s = s0; gb < g1; ++gb) {
        while (a.cu_blocks[s + 1] <= gb) ++s;
        if (a.keep[gb]) {
            const int b = gb - a.cu_blocks[s];
            rows += min(a.G, a.cu_seqlens[s + 1] - a.cu_seqlens[s] - b * a.G);
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
            const int b = gb - a.cu_blocks[s];
            const int len = min(a.G, a.cu_seqlens[s + 1] - a.cu_seqlens[s] - b * a.G);
            a.list[slot++] = make_int4(a.cu_seqlens[s] + b * a.G, dst, len, 0);
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
    const int64_t items = (int64_t)K * a.items_per_block;
    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        const int kb = (int)(it / a.items_per_block);
        const int q = (int)(it % a.items_per_block);
        const int4 e = a.list[kb];  // src row, dst row, rows
        const int r0 = q * a.rows_per_item;
        if (r0 >= e.z) continue;
        const int rows = min(e.z - r0, a.rows_per_item);
        const uint4 *src = a.x + (int64_t)(e.x + r0) * a.vec_per_row;
        uint4 *dst = a.x_out + (int64_t)(e.y + r0) * a.vec_per_row;
        const int64_t nv = (int64_t)rows * a.vec_per_row;
        int64_t v = threadIdx.x;
        for (; v + 3 * kGatherThreads < nv; v += 4 * kGatherThreads) {
            const uint4 x0 = __ldcs(src + v);
            const uint4 x1 = __ldcs(src + v + kGatherThreads);
            const uint4 x2 = __ldcs(src + v + 2 * kGatherThreads);
            const uint4 x3 = __ldcs(src + v + 3 * kGatherThreads);
            __stcs(dst + v, x0);
            __stcs(dst + v + kGatherThreads, x1);
            __stcs(dst + v + 2 * kGatherThreads, x2);
            __stcs(dst + v + 3 * kGatherThreads, x3);
        }
        for (; v < nv; v += kGatherThreads) __stcs(dst + v, __ldcs(src + v));
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
        int lo = 0, hi = B - 1;  // the sequence holding g0
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (cu_blocks[mid] <= g0) lo = mid; else hi = mid - 1;
        }
        int pos = first;
        for (int gb = g0, s = lo; gb < g1; ++gb) {
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
