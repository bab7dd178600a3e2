// select.cu -- top-p block selection, one CTA per sequence.
//
// UniPrefill overview, top-p selection paragraph: sort the blocks by score and
// keep them until the cumulative sum reaches p.  The ranking key packs the
// score's bits (descending) above the block index (ascending) into one 64-bit
// word, so ascending key order is the rank order with ties broken by the lower
// block index.  The block at rank r is kept iff the mass ranked before it is
// < p: that is exactly the shortest prefix whose cumulative mass reaches p
// (crossing block included), and it keeps every block when the total falls
// short of p.  Cumulative masses are exact sums of the fp32 scores in 64-bit
// fixed point (2^-62 resolution), so they do not depend on summation order.
//
// The bitonic sort keeps E consecutive keys per thread in registers: exchanges
// inside a thread use registers, exchanges inside a warp use shuffles, and only
// exchanges across warps go through shared memory.
#include "../../include/up.h"
#include "common.cuh"

namespace up {

namespace {

constexpr int kSelThreads = 1024;
constexpr double kFix = 4611686018427387904.0;  // 2^62

__device__ __forceinline__ unsigned long long rank_key(float score, int idx) {
    // scores are >= 0; -0 and anything not > 0 rank as 0
    const unsigned bits = score > 0.f ? __float_as_uint(score) : 0u;
    return ((unsigned long long)(0xFFFFFFFFu - bits) << 32) | (unsigned)idx;
}

// score * 2^62, truncated (exact for scores >= 2^-38)
__device__ __forceinline__ long long key_fixed(unsigned long long key) {
    const float s = __uint_as_float(0xFFFFFFFFu - (unsigned)(key >> 32));
    return (long long)((double)s * kFix);
}

// compare-exchange for element e against its partner's key b (partner index
// e ^ j): the lower index of the pair keeps min for ascending runs (e & k == 0)
__device__ __forceinline__ unsigned long long cx(unsigned long long a, unsigned long long b, int e,
                                                 int j, int k) {
    const bool lower = (e & j) == 0;
    const bool asc = (e & k) == 0;
    const unsigned long long mn = a < b ? a : b, mx = a < b ? b : a;
    return (lower == asc) ? mn : mx;
}

template <int E>
__device__ __forceinline__ void exchange_in_thread(unsigned long long (&v)[E], int t, int j, int k) {
#pragma unroll
    for (int jj = E / 2; jj >= 1; jj >>= 1) {
        if (j == jj) {
#pragma unroll
            for (int i = 0; i < E; ++i) {
                if ((i & jj) == 0) {
                    const int e = t * E + i;
                    const bool asc = (e & k) == 0;
                    const unsigned long long a = v[i], b = v[i + jj];
                    const bool sw = (a > b) == asc;
                    v[i] = sw ? b : a;
                    v[i + jj] = sw ? a : b;
                }
            }
        }
    }
}

template <int E>
__device__ void bitonic_sort(unsigned long long (&v)[E], int N, unsigned long long *sm) {
    const int t = threadIdx.x;
    for (int k = 2; k <= N; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            if (j >= 32 * E) {
#pragma unroll
                for (int i = 0; i < E; ++i) sm[t * E + i] = v[i];
                __syncthreads();
#pragma unroll
                for (int i = 0; i < E; ++i) {
                    const int e = t * E + i;
                    v[i] = cx(v[i], sm[e ^ j], e, j, k);
                }
                __syncthreads();
            } else if (j >= E) {
                const int m = j / E;  // partner lane
#pragma unroll
                for (int i = 0; i < E; ++i) {
                    const int e = t * E + i;
                    v[i] = cx(v[i], __shfl_xor_sync(0xffffffffu, v[i], m), e, j, k);
                }
            } else {
                exchange_in_thread<E>(v, t, j, k);
            }
        }
    }
}

__device__ long long block_excl_scan_i64(long long v, long long *sh) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[wid] = x;
    __syncthreads();
    if (wid == 0) {
        long long w = sh[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        sh[lane] = w;
    }
    __syncthreads();
    const long long base = wid ? sh[wid - 1] : 0;
    __syncthreads();
    return base + (x - v);
}

template <int E>
__device__ void select_one(const float *__restrict__ scores, int b0, int nb, int N, int L, int G,
                           double p, uint8_t *__restrict__ keep, int32_t *kept_tokens, int s,
                           unsigned long long *sm, long long *shl, int *shi) {
    const int t = threadIdx.x;
    unsigned long long v[E];
#pragma unroll
    for (int i = 0; i < E; ++i) {
        const int e = t * E + i;
        v[i] = e < nb ? rank_key(scores[b0 + e], e) : ~0ull;
    }
    bitonic_sort<E>(v, N, sm);
    // thread t now holds ranks t*E .. t*E+E-1
    long long fx[E], local = 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
        fx[i] = (t * E + i < nb) ? key_fixed(v[i]) : 0;
        local += fx[i];
    }
    long long before = block_excl_scan_i64(local, shl);
    const bool all = !(p < 1.0);
    const long long pfix = all ? 0 : (long long)ceil(p * kFix);
    int kept = 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
        const int r = t * E + i;
        if (r < nb) {
            const int idx = (int)(v[i] & 0xFFFFFFFFull);
            const int k = (all || before < pfix) ? 1 : 0;
            keep[b0 + idx] = (uint8_t)k;
            if (k) kept += min(G, L - idx * G);
        }
        before += fx[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) kept += __shfl_xor_sync(0xffffffffu, kept, o);
    if ((t & 31) == 0) shi[t >> 5] = kept;
    __syncthreads();
    if (t < 32) {
        int w = shi[t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
        if (t == 0) kept_tokens[s] = w;
    }
}

__global__ void __launch_bounds__(kSelThreads)
select_topp_kernel(const float *__restrict__ scores, const int32_t *__restrict__ cu_blocks,
                   const int32_t *__restrict__ cu, int G, double p, uint8_t *__restrict__ keep,
                   int32_t *__restrict__ kept_tokens, unsigned int *err) {
    extern __shared__ unsigned long long sm[];  // [UP_SELECT_MAX_BLOCKS]
    __shared__ long long shl[32];
    __shared__ int shi[32];
    const int s = blockIdx.x;
    const int b0 = cu_blocks[s];
    const int nb = cu_blocks[s + 1] - b0;
    const int L = cu[s + 1] - cu[s];
    if (nb <= 0) {
        if (threadIdx.x == 0) kept_tokens[s] = 0;
        return;
    }
    if (nb > UP_SELECT_MAX_BLOCKS) {
        if (threadIdx.x == 0) {
            atomicOr(err, UP_DEVERR_SELECT_TOO_MANY_BLOCKS);
            kept_tokens[s] = 0;
        }
        return;
    }
    int N = kSelThreads;
    while (N < nb) N <<= 1;
    switch (N / kSelThreads) {
        case 1: select_one<1>(scores, b0, nb, N, L, G, p, keep, kept_tokens, s, sm, shl, shi); break;
        case 2: select_one<2>(scores, b0, nb, N, L, G, p, keep, kept_tokens, s, sm, shl, shi); break;
        case 4: select_one<4>(scores, b0, nb, N, L, G, p, keep, kept_tokens, s, sm, shl, shi); break;
        case 8: select_one<8>(scores, b0, nb, N, L, G, p, keep, kept_tokens, s, sm, shl, shi); break;
        default: select_one<16>(scores, b0, nb, N, L, G, p, keep, kept_tokens, s, sm, shl, shi); break;
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
