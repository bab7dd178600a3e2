// score_fallback.cu -- the exact fallback of block scoring, for the rare row
// tiles whose fp32 sums overflowed in the tensor-core kernel.
//
// The tensor-core kernel measures every partial sum against a reference taken
// from the first 32 keys of a work unit.  If a later key of the same unit has a
// logit more than ~115 binary orders of magnitude above that reference, its
// fp32 sums overflow; the kernel then queues that 128-row tile here (and its
// own epilogue stops: the scores it would write are replaced below).  The
// queue is empty for ordinary attention logits, and this kernel then returns
// at once.
//
// Tiles.  Each queued tile is recomputed with two passes over the logits: the
// first finds each row's exact maximum m over the unit's keys (log2 units),
// the second sums 2^(z*log2e/sqrt(d) - m) over every block.
//
// Rows, then blocks (by the CTA that finishes its tiles last, a counter the
// plan kernel zeroes).  Per row r of a sequence, over its key chunks c:
//     m_r = max_c mref[c][r],  l_r = sum_c lsum[c][r] * 2^(mref[c][r] - m_r),
//     inv_r = 1 / (l_r * n_s * Hq_norm)   (the softmax normaliser and the query/head
//                                         mean; Hq_norm = Hq unless the heads are sharded)
// and then, in place of mref[c][r], the weight of chunk c's partial sums,
//     w[c][r] = 2^(mref[c][r] - m_r) * inv_r;
// finally score_b = sum_r part[b][r] * w[c(b)][r] in a fixed order.  One CTA
// does all rows and blocks: slow, but only taken for overflowing inputs.
// Source: UniPrefill overview, block-wise importance estimation paragraph.
#include "common.cuh"

namespace up {

namespace {

constexpr int kKeyTile = 32;

template <int D>
__device__ __forceinline__ void tile_logits(const __nv_bfloat16 *qT, const float *ks, int tid,
                                            float (&acc)[kKeyTile]) {
#pragma unroll
    for (int kk = 0; kk < kKeyTile; ++kk) acc[kk] = 0.f;
    for (int c = 0; c < D; ++c) {
        const float qv = __bfloat162float(qT[c * kRowsPerTile + tid]);
#pragma unroll
        for (int kk = 0; kk < kKeyTile; ++kk) acc[kk] = fmaf(qv, ks[kk * D + c], acc[kk]);
    }
}

// Rows: a pass takes 64 consecutive rows, lane l holding rows l and l + 32;
// the four warps take every fourth chunk slot and merge (max, sum) online, then
// warp 0 merges the four partial results in warp order -- a fixed order, so the
// result is bitwise reproducible.  The first kCached chunk maxima of each
// (row, warp) stay in registers for the weight pass.
constexpr int kRowsPerPass = 64;
constexpr int kSlotLanes = kRowsPerTile / 32;
constexpr int kCached = 8;

__device__ __forceinline__ void merge_ms(float &m, float &l, float mc, float lc) {
    if (mc == -INFINITY) return;
    if (m == -INFINITY) { m = mc; l = lc; return; }
    const float mn = fmaxf(m, mc);
    l = l * exp2f(m - mn) + lc * exp2f(mc - mn);
    m = mn;
}

__device__ __forceinline__ int find_seq_by_row(const SeqInfo *seqs, int B, int64_t r) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (seqs[mid].row_off <= r) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ float chunk_weight(float mc, float M, float inv) {
    return (mc == -INFINITY || inv == 0.f) ? 0.f : exp2f(mc - M) * inv;
}

// Every pass of CTAs cta, cta + ncta, ... over the `total` rows.  Loads go
// through L2 (.cg): in the queued case they read what other CTAs of this
// kernel wrote.
__device__ __forceinline__ void finalize_rows(const ScoreParams &p, int64_t total, int cta,
                                              int ncta) {
    __shared__ float sm[kSlotLanes][kRowsPerPass], sl[kSlotLanes][kRowsPerPass];
    __shared__ float sM[kRowsPerPass], sI[kRowsPerPass];
    __shared__ int sR[kRowsPerPass];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int64_t g0 = (int64_t)cta * kRowsPerPass; g0 < total;
         g0 += (int64_t)ncta * kRowsPerPass) {
        int nsl[2], R[2];
        float *mr[2];
        const float *ls[2];
        float m[2], l[2], mc[2][kCached];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t gr = g0 + lane + 32 * h;
            const bool ok = gr < total;
            const SeqInfo &sq = p.seqs[find_seq_by_row(p.seqs, p.num_seqs, ok ? gr : total - 1)];
            const int64_t r = (ok ? gr : total - 1) - sq.row_off;
            nsl[h] = ok ? sq.nchunks * kSlotsPerChunk : 0;
            R[h] = sq.R;
            mr[h] = p.mref + sq.stat_off + r;
            ls[h] = p.lsum + sq.stat_off + r;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            m[h] = -INFINITY;
            l[h] = 0.f;
            float lc[kCached];
#pragma unroll
            for (int i = 0; i < kCached; ++i) {
                const int c = wid + kSlotLanes * i;
                mc[h][i] = c < nsl[h] ? __ldcg(mr[h] + (int64_t)c * R[h]) : -INFINITY;
                lc[i] = c < nsl[h] ? __ldcg(ls[h] + (int64_t)c * R[h]) : 0.f;
            }
#pragma unroll
            for (int i = 0; i < kCached; ++i) merge_ms(m[h], l[h], mc[h][i], lc[i]);
            for (int c = wid + kSlotLanes * kCached; c < nsl[h]; c += kSlotLanes)
                merge_ms(m[h], l[h], __ldcg(mr[h] + (int64_t)c * R[h]),
                         __ldcg(ls[h] + (int64_t)c * R[h]));
            sm[wid][lane + 32 * h] = m[h];
            sl[wid][lane + 32 * h] = l[h];
            // the mean over heads divides by n_s * Hq_norm (R = n_s * Hq)
            if (wid == 0) sR[lane + 32 * h] = R[h] / p.Hq * p.Hq_norm;
        }
        __syncthreads();
        if (wid < 2) {
            const int i = lane + 32 * wid;
            float M = sm[0][i], Lsum = sl[0][i];
#pragma unroll
            for (int w = 1; w < kSlotLanes; ++w) merge_ms(M, Lsum, sm[w][i], sl[w][i]);
            sM[i] = M;
            // rows past the total have no chunks: M = -inf, inv 0, nothing written
            sI[i] = (M == -INFINITY || !(Lsum > 0.f)) ? 0.f : 1.0f / (Lsum * (float)sR[i]);
        }
        __syncthreads();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float M = sM[lane + 32 * h], inv = sI[lane + 32 * h];
#pragma unroll
            for (int i = 0; i < kCached; ++i) {
                const int c = wid + kSlotLanes * i;
                if (c < nsl[h]) mr[h][(int64_t)c * R[h]] = chunk_weight(mc[h][i], M, inv);
            }
            for (int c = wid + kSlotLanes * kCached; c < nsl[h]; c += kSlotLanes) {
                float *q = mr[h] + (int64_t)c * R[h];
                *q = chunk_weight(__ldcg(q), M, inv);
            }
        }
        __syncthreads();
    }
}

// Every block score, by one CTA: thread t sums rows t, t + 128, ... of the
// block in order, then a fixed butterfly and the warps in order.
__device__ void finalize_blocks_one_cta(const ScoreParams &p) {
    __shared__ float red[kRowsPerTile / 32];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int nbt = p.counters->blocks;
    int s = 0;
    for (int gb = 0; gb < nbt; ++gb) {
        while (gb >= p.seqs[s].blk_off + p.seqs[s].nb) ++s;  // skips empty sequences
        const SeqInfo &sq = p.seqs[s];
        const int b = gb - sq.blk_off;
        const float *w = p.mref + sq.stat_off + (int64_t)block_slot(b, p.G, p.C) * sq.R;
        const float *pt = p.part + sq.part_off + (int64_t)b * sq.R;
        float acc = 0.f;
        for (int r = threadIdx.x; r < sq.R; r += kRowsPerTile)
            acc = fmaf(__ldcg(pt + r), __ldcg(w + r), acc);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) red[wid] = acc;
        __syncthreads();
        if (threadIdx.x == 0) {
            float t = 0.f;
#pragma unroll
            for (int k = 0; k < kRowsPerTile / 32; ++k) t += red[k];
            p.scores[gb] = t;
        }
        __syncthreads();
    }
}

template <int D>
__global__ void __launch_bounds__(kRowsPerTile, 4)
score_finish_kernel(ScoreParams p) {
    pdl_wait();
    const int nflag = min(p.counters->flagged, p.flag_cap);
    const int64_t total_rows = p.counters->rows;
    if (nflag == 0) return;  // the tensor-core kernel's epilogue wrote the scores
    extern __shared__ __align__(16) unsigned char smem[];
    __nv_bfloat16 *qT = reinterpret_cast<__nv_bfloat16 *>(smem);                 // [D][128]
    float *ks = reinterpret_cast<float *>(smem + D * kRowsPerTile * 2);          // [32][D]
    const int tid = threadIdx.x;
    for (int fi = blockIdx.x; fi < nflag; fi += gridDim.x) {
        const int entry = p.flag_list[fi];
        const int u = entry >> 2;  // work unit; low two bits: which of its row tiles
        const int s = find_seq_by_unit(p.seqs, p.num_seqs, u);
        const SeqInfo sq = p.seqs[s];
        int loc = u - sq.unit_off;
        const int mt = (loc % sq.mtiles) * tiles_per_unit(D) + (entry & 3);
        loc /= sq.mtiles;
        const int c = loc % sq.nchunks;
        const int j = loc / sq.nchunks;

        const int grows = p.g * sq.ns;
        // row tid of the tile: query t = mt * tpt + tid / g of query head j * g + h
        const int tl = tid / p.g, h = tid - tl * p.g;
        const int t = mt * p.tpt + tl;
        const bool valid = tid < p.g * p.tpt && t < sq.ns;
        const int a = sq.L - sq.ns + (valid ? t : 0);
        const int64_t r = (int64_t)j * grows + (int64_t)t * p.g + h;

        __syncthreads();
        for (int idx = tid; idx < kRowsPerTile * D; idx += kRowsPerTile) {
            const int row = idx / D, cc = idx % D;
            const int rtl = row / p.g, rh = row - rtl * p.g, rt = mt * p.tpt + rtl;
            __nv_bfloat16 v = __float2bfloat16(0.f);
            if (row < p.g * p.tpt && rt < sq.ns)
                v = p.q[((int64_t)(sq.q_off + rt) * p.Hq + j * p.g + rh) * D + cc];
            qT[cc * kRowsPerTile + row] = v;
        }

        const int k0 = c * p.C;
        const int k1 = min(k0 + p.C, sq.L);
        float m = -INFINITY;
        float acc[kKeyTile];
        float lsum = 0.f;
        for (int pass = 0; pass < 2; ++pass) {
            float bsum = 0.f;
            for (int kt = k0; kt < k1; kt += kKeyTile) {
                __syncthreads();
                for (int idx = tid; idx < kKeyTile * D; idx += kRowsPerTile) {
                    const int key = kt + idx / D;
                    float v = 0.f;
                    if (key < k1) {
                        if (!p.block_table) {
                            v = __bfloat162float(
                                p.k[((int64_t)(sq.tok_off + key) * p.Hk + j) * D + idx % D]);
                        } else {
                            const int64_t row = paged_row(p, s, j, key);
                            if (row < p.num_pages * p.Hk * p.page_size)
                                v = __bfloat162float(p.k[row * D + idx % D]);
                        }
                    }
                    ks[idx] = v;
                }
                __syncthreads();
                tile_logits<D>(qT, ks, tid, acc);
#pragma unroll
                for (int kk = 0; kk < kKeyTile; ++kk) {
                    const int key = kt + kk;
                    if (key >= k1) break;
                    const bool vis = key <= a;
                    const float z = acc[kk] * p.scale_log2;
                    if (pass == 0) {
                        if (vis) m = fmaxf(m, z);
                    } else {
                        const float e = (vis && m != -INFINITY) ? exp2f(z - m) : 0.f;
                        bsum += e;
                        if ((key + 1) % p.G == 0 || key + 1 == k1) {
                            if (valid) p.part[sq.part_off + (int64_t)(key / p.G) * sq.R + r] = bsum;
                            lsum += bsum;
                            bsum = 0.f;
                        }
                    }
                }
            }
        }
        if (valid) {
            const int64_t o = sq.stat_off + (int64_t)(kSlotsPerChunk * c) * sq.R + r;
            p.mref[o] = m;
            p.lsum[o] = lsum;
        }
    }
    // every CTA's recomputed tiles are in memory before the last one reads them
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(&const_cast<Counters *>(p.counters)->fin_done, 1) == (int)gridDim.x - 1;
    __syncthreads();
    if (s_last) {
        __threadfence();
        finalize_rows(p, total_rows, 0, 1);
        __threadfence();
        __syncthreads();
        finalize_blocks_one_cta(p);
    }
}

template <int D>
cudaError_t launch_d(const ScoreParams &p, int64_t max_rows, int num_sms, cudaStream_t st) {
    const size_t smem = (size_t)D * kRowsPerTile * 2 + (size_t)kKeyTile * D * 4;
    cudaError_t e = cudaFuncSetAttribute(score_finish_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // one CTA per SM for the queue (empty for ordinary inputs: every CTA returns at once)
    (void)max_rows;
    return launch_pdl(score_finish_kernel<D>, dim3(num_sms), dim3(kRowsPerTile), smem, st, p);
}

}  // namespace

cudaError_t launch_score_finish(const ScoreParams &p, const ScoreLayout &lay, int num_sms,
                               cudaStream_t st) {
    switch (p.d) {
        case 64: return launch_d<64>(p, lay.max_rows, num_sms, st);
        case 128: return launch_d<128>(p, lay.max_rows, num_sms, st);
        case 256: return launch_d<256>(p, lay.max_rows, num_sms, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace up
