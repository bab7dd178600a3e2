// score_plan.cu -- work planning and the deterministic finalize of block scoring.
//
// Scoring is split into three steps:
//   plan      (1 CTA)  cu_seqlens -> per-sequence table, cu_blocks, work-unit count.
//   main      (score kernel) per (row, block) partial softmax sums relative to a
//             per (row, chunk) reference, plus the chunk's reference and sum.
//             A work unit is (sequence, KV head, pair of 128-row tiles, key chunk).
//   finalize  rows:   per row, merge the chunk statistics into the row's softmax
//                     normaliser and turn each chunk reference into a weight;
//             blocks: per block, a fixed-order weighted sum over the sequence's
//                     rows -> the block score.
// UniPrefill overview, block-wise importance estimation paragraph: the block
// score is the softmax attention mass of the last n queries that falls into a
// block, averaged over queries and heads (the "online softmax" and "block
// reduction" of its fused-kernel paragraph).
#include "common.cuh"

namespace up {

namespace {

constexpr int kPlanThreads = 1024;

// Block-wide exclusive scan of one int64 per thread (blockDim.x == 1024).
__device__ int64_t block_excl_scan(int64_t v, int64_t *total, int64_t *sh) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int64_t w = sh[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int64_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        sh[lane] = w;  // inclusive prefix of warp totals
    }
    __syncthreads();
    const int64_t warp_base = wid ? sh[wid - 1] : 0;
    *total = sh[31];
    __syncthreads();
    return warp_base + x - v;
}

__global__ void __launch_bounds__(kPlanThreads)
score_plan_kernel(const int32_t *__restrict__ cu, int32_t *__restrict__ cu_blocks,
                  SeqInfo *__restrict__ seqs, Counters *__restrict__ cnt, int B,
                  int64_t total_tokens, int Hq, int Hk, int n, int G, int C,
                  unsigned int *err) {
    __shared__ int64_t sh[32];
    const int g = Hq / Hk;
    // validate cu_seqlens
    int bad = 0;
    for (int s = threadIdx.x; s <= B; s += blockDim.x) {
        const int v = cu[s];
        if (s == 0 && v != 0) bad = 1;
        if (s > 0 && v < cu[s - 1]) bad = 1;
        if (s == B && (int64_t)v != total_tokens) bad = 1;
    }
    bad = __syncthreads_or(bad);
    if (bad) {
        if (threadIdx.x == 0) {
            atomicOr(err, 0x1u);
            cnt->units = 0; cnt->blocks = 0; cnt->rows = 0; cnt->flagged = 0;
        }
        for (int s = threadIdx.x; s <= B; s += blockDim.x) cu_blocks[s] = 0;
        return;
    }
    int64_t base_q = 0, base_b = 0, base_u = 0, base_r = 0, base_p = 0, base_s = 0;
    for (int t0 = 0; t0 < B; t0 += blockDim.x) {
        const int s = t0 + threadIdx.x;
        int64_t L = 0, ns = 0, nb = 0, nch = 0, mt = 0, R = 0, units = 0;
        if (s < B) {
            L = cu[s + 1] - cu[s];
            ns = L < n ? L : n;
            nb = (L + G - 1) / G;
            nch = (L + C - 1) / C;
            mt = (g * ns + kTilesPerUnit * kRowsPerTile - 1) / (kTilesPerUnit * kRowsPerTile);
            R = (int64_t)Hq * ns;
            units = (int64_t)Hk * mt * nch;
        }
        int64_t tq, tb, tu, tr, tp, ts;
        const int64_t oq = block_excl_scan(ns, &tq, sh);
        const int64_t ob = block_excl_scan(nb, &tb, sh);
        const int64_t ou = block_excl_scan(units, &tu, sh);
        const int64_t orow = block_excl_scan(R, &tr, sh);
        const int64_t op = block_excl_scan(R * nb, &tp, sh);
        const int64_t os = block_excl_scan(R * nch * kSlotsPerChunk, &ts, sh);
        if (s < B) {
            SeqInfo si;
            si.tok_off = cu[s];
            si.L = (int32_t)L;
            si.ns = (int32_t)ns;
            si.q_off = (int32_t)(base_q + oq);
            si.nb = (int32_t)nb;
            si.blk_off = (int32_t)(base_b + ob);
            si.nchunks = (int32_t)nch;
            si.mtiles = (int32_t)mt;
            si.R = (int32_t)R;
            si.unit_off = (int32_t)(base_u + ou);
            si.row_off = base_r + orow;
            si.part_off = base_p + op;
            si.stat_off = base_s + os;
            seqs[s] = si;
            cu_blocks[s] = si.blk_off;
        }
        base_q += tq; base_b += tb; base_u += tu; base_r += tr; base_p += tp; base_s += ts;
    }
    if (threadIdx.x == 0) {
        cu_blocks[B] = (int32_t)base_b;
        cnt->units = (int32_t)base_u;
        cnt->blocks = (int32_t)base_b;
        cnt->rows = base_r;
        cnt->flagged = 0;
    }
}

__device__ __forceinline__ int find_seq_by_row(const SeqInfo *seqs, int B, int64_t r) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (seqs[mid].row_off <= r) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ int find_seq_by_block(const SeqInfo *seqs, int B, int b) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (seqs[mid].blk_off <= b) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Per row: m = max_c mref, l = sum_c lsum_c * 2^(mref_c - m), and the weight of
// key chunk c: w_c = 2^(mref_c - m) / (l * R), R = n_s * Hq (the query/head mean).
__global__ void __launch_bounds__(256)
finalize_rows_kernel(ScoreParams p) {
    const int64_t total = p.counters->rows;
    for (int64_t gr = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; gr < total;
         gr += (int64_t)gridDim.x * blockDim.x) {
        const int s = find_seq_by_row(p.seqs, p.num_seqs, gr);
        const SeqInfo sq = p.seqs[s];
        const int64_t r = gr - sq.row_off;
        const float *mr = p.mref + sq.stat_off + r;
        const float *ls = p.lsum + sq.stat_off + r;
        const int nslots = sq.nchunks * kSlotsPerChunk;
        float m = -INFINITY;
        for (int c = 0; c < nslots; ++c) m = fmaxf(m, mr[(int64_t)c * sq.R]);
        float l = 0.f;
        for (int c = 0; c < nslots; ++c) {
            const float mc = mr[(int64_t)c * sq.R];
            if (mc != -INFINITY) l += ls[(int64_t)c * sq.R] * exp2f(mc - m);
        }
        const float inv = 1.0f / (l * (float)sq.R);
        float *w = p.w + sq.stat_off + r;
        for (int c = 0; c < nslots; ++c) {
            const float mc = mr[(int64_t)c * sq.R];
            w[(int64_t)c * sq.R] = (mc == -INFINITY) ? 0.f : exp2f(mc - m) * inv;
        }
    }
}

// One warp per block: score = sum_r w[c(b)][r] * part[b][r], lanes take rows
// lane, lane+32, ... in order, then a fixed butterfly: bitwise reproducible.
__global__ void __launch_bounds__(256)
finalize_blocks_kernel(ScoreParams p) {
    const int total = p.counters->blocks;
    const int lane = threadIdx.x & 31;
    const int warps = (gridDim.x * blockDim.x) >> 5;
    for (int gb = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; gb < total; gb += warps) {
        const int s = find_seq_by_block(p.seqs, p.num_seqs, gb);
        const SeqInfo sq = p.seqs[s];
        const int b = gb - sq.blk_off;
        const int c = block_slot(b, p.G, p.C);
        const float *w = p.w + sq.stat_off + (int64_t)c * sq.R;
        const float *pt = p.part + sq.part_off + (int64_t)b * sq.R;
        float acc = 0.f;
        for (int r = lane; r < sq.R; r += 32) acc = fmaf(__ldg(w + r), __ldcs(pt + r), acc);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) p.scores[gb] = acc;
    }
}

}  // namespace

cudaError_t launch_score_plan(const int32_t *cu_seqlens, int32_t *cu_blocks, const ScoreParams &p,
                              int64_t total_tokens, cudaStream_t st) {
    score_plan_kernel<<<1, kPlanThreads, 0, st>>>(
        cu_seqlens, cu_blocks, const_cast<SeqInfo *>(p.seqs), const_cast<Counters *>(p.counters),
        p.num_seqs, total_tokens, p.Hq, p.Hk, p.n, p.G, p.C, p.err);
    return cudaGetLastError();
}

cudaError_t launch_score_finalize(const ScoreParams &p, const ScoreLayout &lay, cudaStream_t st) {
    if (lay.max_rows > 0) {
        const int64_t want = (lay.max_rows + 255) / 256;
        const int grid = (int)(want < 65535 ? want : 65535);
        finalize_rows_kernel<<<grid, 256, 0, st>>>(p);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (lay.max_blocks > 0) {
        const int64_t want = (lay.max_blocks + 7) / 8;  // 8 warps per CTA
        const int grid = (int)(want < 65535 ? want : 65535);
        finalize_blocks_kernel<<<grid, 256, 0, st>>>(p);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

}  // namespace up
