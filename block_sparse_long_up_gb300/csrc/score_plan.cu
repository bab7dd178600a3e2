// score_plan.cu -- work planning of block scoring.
//
// Scoring runs as
//   plan    (1 warp) cu_seqlens -> per-sequence table, cu_blocks, work-unit
//           count; zeroes the counters of the scoring kernel's grid barriers.
//   main    (tensor-core kernel, score_tc.cu) per (row, block) partial softmax
//           sums relative to a per (row, chunk) reference, the chunk's
//           reference and sum; then, across the whole grid, the exact
//           recomputation of any tile whose sums overflowed, every row's
//           normaliser and chunk weights, and every block score.
// UniPrefill overview, block-wise importance estimation paragraph: the block
// score is the softmax attention mass of the last n queries that falls into a
// block, averaged over queries and heads.
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
            cnt->units = 0; cnt->blocks = 0; cnt->rows = 0; cnt->flagged = 0;
            cnt->bar[0] = 0; cnt->bar[1] = 0; cnt->bar[2] = 0;
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
        cnt->bar[0] = 0;
        cnt->bar[1] = 0;
        cnt->bar[2] = 0;
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

}  // namespace up
