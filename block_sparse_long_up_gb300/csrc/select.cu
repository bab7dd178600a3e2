// select.cu -- top-p block selection, one CTA per sequence.
//
// UniPrefill overview, top-p selection paragraph: sort the blocks by score and
// keep them until the cumulative sum reaches p.  The ranking key packs the
// score's bits (descending) above the block index (ascending) into one 64-bit
// word, so one on-chip bitonic sort gives the order with ties broken by the
// lower block index.  The cumulative sum is an fp64 scan in rank order; the
// cut is the first rank whose inclusive sum is >= p (crossing block kept).
#include "../../include/up.h"
#include "common.cuh"

namespace up {

namespace {

constexpr int kSelThreads = 1024;

__device__ __forceinline__ unsigned long long rank_key(float score, int idx) {
    // scores are >= 0; -0 and anything not > 0 rank as 0
    const unsigned bits = score > 0.f ? __float_as_uint(score) : 0u;
    return ((unsigned long long)(0xFFFFFFFFu - bits) << 32) | (unsigned)idx;
}

__device__ __forceinline__ double key_score(unsigned long long key) {
    return (double)__uint_as_float(0xFFFFFFFFu - (unsigned)(key >> 32));
}

// Block-wide exclusive scan of one double per thread, fixed association order.
__device__ double block_excl_scan_f64(double v, double *sh) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    double x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[wid] = x;
    __syncthreads();
    if (wid == 0) {
        double w = sh[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        sh[lane] = w;
    }
    __syncthreads();
    const double base = wid ? sh[wid - 1] : 0.0;
    __syncthreads();
    return base + (x - v);
}

__global__ void __launch_bounds__(kSelThreads)
select_topp_kernel(const float *__restrict__ scores, const int32_t *__restrict__ cu_blocks,
                   const int32_t *__restrict__ cu, int G, double p, uint8_t *__restrict__ keep,
                   int32_t *__restrict__ kept_tokens, unsigned int *err) {
    extern __shared__ unsigned long long keys[];  // [UP_SELECT_MAX_BLOCKS]
    __shared__ double sh_d[32];
    __shared__ int sh_i[32];
    __shared__ int s_rstar;
    const int s = blockIdx.x, tid = threadIdx.x;
    const int b0 = cu_blocks[s];
    const int nb = cu_blocks[s + 1] - b0;
    const int L = cu[s + 1] - cu[s];
    if (nb <= 0) {
        if (tid == 0) kept_tokens[s] = 0;
        return;
    }
    if (nb > UP_SELECT_MAX_BLOCKS) {
        if (tid == 0) {
            atomicOr(err, UP_DEVERR_SELECT_TOO_MANY_BLOCKS);
            kept_tokens[s] = 0;
        }
        return;
    }
    int N = 1;
    while (N < nb) N <<= 1;
    for (int i = tid; i < N; i += kSelThreads)
        keys[i] = i < nb ? rank_key(scores[b0 + i], i) : ~0ull;
    if (tid == 0) s_rstar = nb - 1;
    __syncthreads();

    // bitonic sort, ascending keys = descending score, ascending index
    for (int k = 2; k <= N; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < (N >> 1); i += kSelThreads) {
                const int lo = ((i & ~(j - 1)) << 1) | (i & (j - 1));
                const int hi = lo + j;
                const bool asc = (lo & k) == 0;
                const unsigned long long x = keys[lo], y = keys[hi];
                if ((x > y) == asc) { keys[lo] = y; keys[hi] = x; }
            }
            __syncthreads();
        }
    }

    // fp64 inclusive scan in rank order: thread tid owns ranks [tid*E, tid*E+E)
    const int E = (N + kSelThreads - 1) / kSelThreads;
    const int beg = tid * E;
    double local = 0.0;
    for (int e = 0; e < E; ++e) {
        const int r = beg + e;
        if (r < nb) local += key_score(keys[r]);
    }
    const double pre = block_excl_scan_f64(local, sh_d);
    if (p < 1.0) {
        double c = pre;
        for (int e = 0; e < E; ++e) {
            const int r = beg + e;
            if (r >= nb) break;
            c += key_score(keys[r]);
            if (c >= p) { atomicMin(&s_rstar, r); break; }
        }
    }
    __syncthreads();
    const int rstar = s_rstar;

    int kept = 0;
    for (int r = tid; r < nb; r += kSelThreads) {
        const int idx = (int)(keys[r] & 0xFFFFFFFFull);
        const int k = r <= rstar;
        keep[b0 + idx] = (uint8_t)k;
        if (k) kept += min(G, L - idx * G);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) kept += __shfl_xor_sync(0xffffffffu, kept, o);
    if ((tid & 31) == 0) sh_i[tid >> 5] = kept;
    __syncthreads();
    if (tid < 32) {
        int v = sh_i[tid];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (tid == 0) kept_tokens[s] = v;
    }
}

}  // namespace

cudaError_t launch_select(const float *scores, const int32_t *cu_blocks, const int32_t *cu_seqlens,
                          int num_seqs, int G, double p, uint8_t *keep, int32_t *kept_tokens,
                          unsigned int *err, cudaStream_t st) {
    const int smem = UP_SELECT_MAX_BLOCKS * (int)sizeof(unsigned long long);
    cudaError_t e = cudaFuncSetAttribute(select_topp_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (num_seqs <= 0) return cudaSuccess;
    select_topp_kernel<<<num_seqs, kSelThreads, smem, st>>>(scores, cu_blocks, cu_seqlens, G, p,
                                                             keep, kept_tokens, err);
    return cudaGetLastError();
}

}  // namespace up
