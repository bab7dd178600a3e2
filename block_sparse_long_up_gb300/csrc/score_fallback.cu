// score_simt.cu -- exact CUDA-core fallback for score work units.
//
// The tensor-core kernel measures every partial sum against a reference taken
// from the first 32 keys of a work unit.  If a later key of the same unit has a
// logit more than ~115 binary orders of magnitude above that reference, its fp32
// sums overflow; the kernel then queues that 128-row tile here.  This kernel
// recomputes such a tile with two passes over the logits: the first finds each
// row's exact maximum m over the unit's keys (log2 units), the second sums
// 2^(z*log2e/sqrt(d) - m) over every block.  The queue is empty for ordinary
// attention logits.
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

template <int D>
__global__ void __launch_bounds__(kRowsPerTile)
score_fallback_kernel(ScoreParams p) {
    pdl_trigger();
    pdl_wait();
    const int nflag = min(p.counters->flagged, p.flag_cap);
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
                    ks[idx] = key < k1 ? __bfloat162float(
                                             p.k[((int64_t)(sq.tok_off + key) * p.Hk + j) * D + idx % D])
                                       : 0.f;
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
}

template <int D>
cudaError_t launch_d(const ScoreParams &p, int num_sms, cudaStream_t st) {
    const size_t smem = (size_t)D * kRowsPerTile * 2 + (size_t)kKeyTile * D * 4;
    cudaError_t e = cudaFuncSetAttribute(score_fallback_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(score_fallback_kernel<D>, dim3(num_sms), dim3(kRowsPerTile), smem, st, p);
}

}  // namespace

cudaError_t launch_score_fallback(const ScoreParams &p, int num_sms, cudaStream_t st) {
    switch (p.d) {
        case 64: return launch_d<64>(p, num_sms, st);
        case 128: return launch_d<128>(p, num_sms, st);
        case 256: return launch_d<256>(p, num_sms, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace up
