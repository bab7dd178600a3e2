// score_plan.cu -- work planning and the deterministic finalize of block scoring.
//
// Scoring is split into three steps:
//   plan      (1 warp) cu_seqlens -> per-sequence table, cu_blocks, work-unit count.
//   main      (score kernel) per (row, block) partial softmax sums relative to a
//             per (row, chunk) reference, plus the chunk's reference and sum.
//             A work unit is (sequence, KV head, group of 128-row tiles, key chunk).
//   finalize  rows:   per row, merge the chunk statistics into the row's softmax
//                     maximum and normaliser;
//             blocks: per block, a fixed-order weighted sum over the sequence's
//                     rows (weight of a partial = 2^(chunk ref - row max) /
//                     (normaliser * rows)) -> the block score.
// UniPrefill overview, block-wise importance estimation paragraph: the block
// score is the softmax attention mass of the last n queries that falls into a
// block, averaged over queries and heads (the "online softmax" and "block
// reduction" of its fused-kernel paragraph).
#include "common.cuh"

namespace up {

namespace {

constexpr int kPlanThreads = 32;  // one warp: shuffle scans, no block barriers

// Warp-wide exclusive scan of one int64 per lane; *total = sum over the warp.
__device__ __forceinline__ int64_t warp_excl_scan(int64_t v, int64_t *total) {
    const int lane = threadIdx.x & 31;
    int64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    *total = __shfl_sync(0xffffffffu, x, 31);
    return x - v;
}

// The plan: one warp walks the sequences 32 at a time (lane = sequence) and
// carries the running offsets from one group to the next.
__global__ void __launch_bounds__(kPlanThreads)
score_plan_kernel(const int32_t *__restrict__ cu, int32_t *__restrict__ cu_blocks,
                  SeqInfo *__restrict__ seqs, Counters *__restrict__ cnt, int B,
                  int64_t total_tokens, int Hq, int Hk, int d, int n, int G, int C,
                  int page_size, int max_pages, unsigned int *err) {
    pdl_wait();
    pdl_trigger();  // after the wait: every kernel before this one is complete
    const int lane = threadIdx.x;
    const int g = Hq / Hk;
    // validate cu_seqlens
    int bad = 0;
    for (int s = lane; s <= B; s += 32) {
        const int v = cu[s];
        if (s == 0 && v != 0) bad = 1;
        if (s > 0 && v < cu[s - 1]) bad = 1;
        if (s == B && (int64_t)v != total_tokens) bad = 1;
        // paged keys: every sequence fits its block-table row
        if (s > 0 && page_size > 0 && v >= cu[s - 1] &&
            (int64_t)(v - cu[s - 1] + page_size - 1) / page_size > max_pages)
            bad = 1;
    }
    if (__any_sync(0xffffffffu, bad)) {
        // leave a well-formed empty plan: every later kernel sees no work
        if (lane == 0) {
            atomicOr(err, 0x1u);
            cnt->units = 0; cnt->blocks = 0; cnt->rows = 0; cnt->flagged = 0; cnt->fin_done = 0;
        }
        for (int s = lane; s <= B; s += 32) {
            cu_blocks[s] = 0;
            if (s < B) seqs[s] = SeqInfo{};
        }
        return;
    }
    int64_t base_q = 0, base_b = 0, base_u = 0, base_r = 0, base_p = 0, base_s = 0;
    for (int t0 = 0; t0 < B; t0 += 32) {
        const int s = t0 + lane;
        int64_t L = 0, ns = 0, nb = 0, nch = 0, mt = 0, R = 0, units = 0;
        if (s < B) {
            L = cu[s + 1] - cu[s];
            ns = L < n ? L : n;
            nb = (L + G - 1) / G;
            nch = (L + C - 1) / C;
            const int64_t tpt = tokens_per_tile(g), tpu = tiles_per_unit(d);
            mt = ((ns + tpt - 1) / tpt + tpu - 1) / tpu;
            R = (int64_t)Hq * ns;
            units = (int64_t)Hk * mt * nch;
        }
        int64_t tq, tb, tu, tr, tp, ts;
        const int64_t oq = warp_excl_scan(ns, &tq);
        const int64_t ob = warp_excl_scan(nb, &tb);
        const int64_t ou = warp_excl_scan(units, &tu);
        const int64_t orow = warp_excl_scan(R, &tr);
        const int64_t op = warp_excl_scan(R * nb, &tp);
        const int64_t os = warp_excl_scan(R * nch * kSlotsPerChunk, &ts);
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
    if (lane == 0) {
        cu_blocks[B] = (int32_t)base_b;
        cnt->units = (int32_t)base_u;
        cnt->blocks = (int32_t)base_b;
        cnt->rows = base_r;
        cnt->flagged = 0;
        cnt->fin_done = 0;
    }
}

// Block scores.  score_b = sum_r part[b][r] * w[c(b)][r], with c(b) the chunk
// of block b.  A CTA takes a contiguous run of the blocks and walks it in
// batches of up to kFinBatch blocks of one sequence and one chunk: a batch
// shares one weight row, read once (the next batch of the same chunk finds it
// in L1), and all of its partials are in flight together.  Thread t takes the
// float4 groups t, t + 256, t + 512, ... of the rows, in increasing order, into
// one accumulator per block; a fixed butterfly and the eight warps in order
// finish the sum.  The order depends neither on the grid nor on the batching,
// so the result is bitwise reproducible.
constexpr int kFinThreads = 256;
constexpr int kFinWarps = kFinThreads / 32;
constexpr int kFinBatch = 4;      // blocks per batch
constexpr int kFinUnroll = 4;     // float4 groups per thread and block in flight
constexpr int kFinCtasPerSm = 4;

// 16-byte loads: streaming (partials, read once) and read-only cached (weights).
__device__ __forceinline__ float4 ld_stream4(const float4 *p) {
    float4 v;
    asm volatile("ld.global.cs.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ float4 ld_ro4(const float4 *p) {
    float4 v;
    asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float dot4(const float4 x, const float4 y, float a) {
    a = fmaf(x.x, y.x, a);
    a = fmaf(x.y, y.y, a);
    a = fmaf(x.z, y.z, a);
    return fmaf(x.w, y.w, a);
}

__device__ __forceinline__ int find_seq_by_block(const SeqInfo *seqs, int B, int gb) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (seqs[mid].blk_off <= gb) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__global__ void __launch_bounds__(kFinThreads) finalize_blocks_kernel(ScoreParams p) {
    __shared__ float red[2][kFinBatch][kFinWarps];
    pdl_wait();
    const int nbt = p.counters->blocks;  // 0 when the plan is invalid
    const int per = (nbt + (int)gridDim.x - 1) / (int)gridDim.x;
    const int lo = (int)blockIdx.x * per, hi = min(lo + per, nbt);
    if (lo >= hi) return;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int bpc = p.C / p.G;  // blocks per key chunk
    int s = find_seq_by_block(p.seqs, p.num_seqs, lo);
    SeqInfo sq = p.seqs[s];
    int par = 0;
    for (int gb = lo; gb < hi; par ^= 1) {
        while (gb >= sq.blk_off + sq.nb) sq = p.seqs[++s];  // skips empty sequences
        const int b = gb - sq.blk_off;
        const int nbat = min(min(kFinBatch, hi - gb), min(sq.nb - b, (b / bpc + 1) * bpc - b));
        const float *wr = p.mref + sq.stat_off + (int64_t)block_slot(b, p.G, p.C) * sq.R;
        const float *pt = p.part + sq.part_off + (int64_t)b * sq.R;
        float acc[kFinBatch];
#pragma unroll
        for (int k = 0; k < kFinBatch; ++k) acc[k] = 0.f;
        if ((sq.R % 4 == 0) && ((reinterpret_cast<uintptr_t>(wr) & 15) == 0) &&
            ((reinterpret_cast<uintptr_t>(pt) & 15) == 0)) {
            const float4 *w4 = reinterpret_cast<const float4 *>(wr);
            const float4 *p4 = reinterpret_cast<const float4 *>(pt);
            const int R4 = sq.R / 4;
            const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int i0 = threadIdx.x; i0 < R4; i0 += kFinUnroll * kFinThreads) {
                float4 w[kFinUnroll], x[kFinBatch][kFinUnroll];
#pragma unroll
                for (int u = 0; u < kFinUnroll; ++u) {
                    const int i = i0 + u * kFinThreads;
                    w[u] = i < R4 ? ld_ro4(w4 + i) : zero;
                }
#pragma unroll
                for (int k = 0; k < kFinBatch; ++k)
#pragma unroll
                    for (int u = 0; u < kFinUnroll; ++u) {
                        const int i = i0 + u * kFinThreads;
                        x[k][u] = (k < nbat && i < R4) ? ld_stream4(p4 + (int64_t)k * R4 + i)
                                                       : zero;
                    }
#pragma unroll
                for (int k = 0; k < kFinBatch; ++k)
#pragma unroll
                    for (int u = 0; u < kFinUnroll; ++u) acc[k] = dot4(x[k][u], w[u], acc[k]);
            }
        } else {
            for (int r = threadIdx.x; r < sq.R; r += kFinThreads) {
                const float w = __ldg(wr + r);
#pragma unroll
                for (int k = 0; k < kFinBatch; ++k)
                    if (k < nbat) acc[k] = fmaf(__ldcs(pt + (int64_t)k * sq.R + r), w, acc[k]);
            }
        }
#pragma unroll
        for (int k = 0; k < kFinBatch; ++k) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], o);
        }
        if (lane == 0) {
#pragma unroll
            for (int k = 0; k < kFinBatch; ++k) red[par][k][wid] = acc[k];
        }
        // one barrier per batch: red is double-buffered, and a buffer is written
        // again only after the next batch's barrier, which its readers reach
        // after reading it
        __syncthreads();
        if ((int)threadIdx.x < nbat) {
            const float *rq = red[par][threadIdx.x];
            float t = 0.f;
#pragma unroll
            for (int w = 0; w < kFinWarps; ++w) t += rq[w];
            p.scores[gb + threadIdx.x] = t;
        }
        gb += nbat;
    }
}

}  // namespace

cudaError_t launch_score_plan(const int32_t *cu_seqlens, int32_t *cu_blocks, const ScoreParams &p,
                              int64_t total_tokens, cudaStream_t st) {
    return launch_pdl(score_plan_kernel, dim3(1), dim3(kPlanThreads), 0, st, cu_seqlens, cu_blocks,
                      const_cast<SeqInfo *>(p.seqs), const_cast<Counters *>(p.counters),
                      p.num_seqs, total_tokens, p.Hq, p.Hk, p.d, p.n, p.G, p.C,
                      p.block_table ? p.page_size : 0, p.max_pages, p.err);
}

cudaError_t launch_score_finalize(const ScoreParams &p, const ScoreLayout &lay, int num_sms,
                                  cudaStream_t st) {
    if (lay.max_blocks <= 0) return cudaSuccess;
    // a contiguous run of blocks per CTA (CTAs past the real block count exit at once)
    const int64_t cap = (int64_t)kFinCtasPerSm * num_sms;
    const int grid = (int)(lay.max_blocks < cap ? lay.max_blocks : cap);
    return launch_pdl(finalize_blocks_kernel, dim3(grid), dim3(kFinThreads), 0, st, p);
}

}  // namespace up
