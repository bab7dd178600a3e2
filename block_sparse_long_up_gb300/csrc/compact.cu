// compact.cu -- gather the kept tokens' hidden states and positions.
//
// UniPrefill overview, sparsity-propagation paragraph: every later sub-layer
// takes only the kept tokens; system-integration paragraph: the kept tokens'
// positions travel with them.  A kept block is a contiguous run of at most G
// rows, so compaction is a set of contiguous copies:
//   index  (1 CTA)  exclusive scans over all blocks -> kept-block list
//                   (source row, destination row, rows), cu_seqlens_out, total;
//   gather (persistent grid) one work item = up to rows_per_item rows of one
//                   kept block, copied with 16-byte vector loads and stores.
#include "common.cuh"

namespace up {

namespace {

constexpr int kIndexThreads = 1024;
constexpr int kGatherThreads = 512;

__device__ int block_excl_scan_i32(int v, int *total, int *sh) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int w = sh[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        sh[lane] = w;
    }
    __syncthreads();
    const int base = wid ? sh[wid - 1] : 0;
    *total = sh[31];
    __syncthreads();
    return base + x - v;
}

__global__ void __launch_bounds__(kIndexThreads)
compact_index_kernel(CompactArgs a) {
    pdl_trigger();
    pdl_wait();
    int32_t *dst_blk = a.dst_blk;
    __shared__ int sh[32];
    const int B = a.num_seqs;
    const int total_blocks = a.cu_blocks[B];
    int carry_rows = 0, carry_k = 0;
    for (int t0 = 0; t0 < total_blocks; t0 += kIndexThreads) {
        const int gb = t0 + threadIdx.x;
        int len = 0, kf = 0, src = 0;
        if (gb < total_blocks) {
            int lo = 0, hi = B - 1;  // last sequence whose first block is <= gb
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (a.cu_blocks[mid] <= gb) lo = mid; else hi = mid - 1;
            }
            const int b = gb - a.cu_blocks[lo];
            const int L = a.cu_seqlens[lo + 1] - a.cu_seqlens[lo];
            src = a.cu_seqlens[lo] + b * a.G;
            if (a.keep[gb]) {
                len = min(a.G, L - b * a.G);
                kf = 1;
            }
        }
        int tot_rows, tot_k;
        const int er = block_excl_scan_i32(len, &tot_rows, sh);
        const int ek = block_excl_scan_i32(kf, &tot_k, sh);
        if (gb < total_blocks) {
            dst_blk[gb] = carry_rows + er;
            if (kf) a.list[carry_k + ek] = make_int4(src, carry_rows + er, len, 0);
        }
        carry_rows += tot_rows;
        carry_k += tot_k;
    }
    __syncthreads();
    for (int s = threadIdx.x; s <= B; s += kIndexThreads) {
        const int cb = a.cu_blocks[s];
        a.cu_out[s] = cb < total_blocks ? dst_blk[cb] : carry_rows;
    }
    if (threadIdx.x == 0) {
        *a.total_kept = carry_rows;
        *a.nkept = carry_k;
    }
}

__global__ void __launch_bounds__(kGatherThreads)
compact_gather_kernel(CompactArgs a) {
    pdl_trigger();
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

}  // namespace

cudaError_t launch_compact(const CompactArgs &a, int num_sms, cudaStream_t st) {
    cudaError_t e = launch_pdl(compact_index_kernel, dim3(1), dim3(kIndexThreads), 0, st, a);
    if (e != cudaSuccess) return e;
    return launch_pdl(compact_gather_kernel, dim3(num_sms * 4), dim3(kGatherThreads), 0, st, a);
}

}  // namespace up
