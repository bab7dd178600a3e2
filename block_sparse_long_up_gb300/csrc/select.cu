// select.cu -- top-p (and top-k) block selection, one CTA per sequence.
//
// UniPrefill overview, top-p selection paragraph: sort the blocks by score and
// keep them until the cumulative sum reaches p.  The ranking key packs the
// score's bits (descending) above the block index (ascending) into one 64-bit
// word, so ascending key order is the rank order with ties broken by the lower
// block index.  The block at rank r is kept iff the mass ranked before it is
// < p: that is exactly the shortest prefix whose cumulative mass reaches p
// (crossing block included), and it keeps every block when the total falls
// short of p.  Masses are the fp32 scores in 64-bit fixed point (score * 2^62,
// truncated, by integer shifts of the float's fields), so every cumulative mass
// is an exact integer sum that does not depend on summation order.
//
// Top-k (UniPrefill overview, hyper-parameters paragraph: the ablation against
// a fixed number of kept blocks) is the same search with every key's mass set
// to 1 and P = k: the block at rank r is kept iff r < k.  The keep-last option
// (after either rule) also keeps each sequence's last block.
//
// No sort is needed: the kept set is {key <= K*} for K*, the last key whose
// mass-before is < P (top-p: P = ceil(p * 2^62)).  K* is found digit by digit,
// most significant first.  A pass histograms the exact masses and counts of
// the keys that share the digits found so far over their next digit (4096
// buckets in shared memory, exact 64-bit sums), one CTA-wide scan gives every
// bucket its mass-before, and the last non-empty bucket whose mass-before is
// < P holds K* (its first key is kept, the first key of any later bucket is
// not).  The first digit is the score's exponent and top four mantissa bits,
// so at ordinary score distributions one pass leaves a few keys in that bucket;
// as soon as at most kSmallM remain, each of them takes its exact mass-before
// by comparing itself with the others.  Ties (equal scores) are separated by
// the index digits.  Five passes at most: score bits 30..19, 18..7, 6..0, then
// index bits 15..4 and 3..0.
//
// Before the passes, one CTA-wide reduction gives the masses (and counts) of
// the keys with scores >= 2^-8, >= 2^-14 and >= 2^-20 (a sequence's scores sum
// to 1).  If the keys at or above such a threshold already hold mass >= P,
// every key below it has mass-before >= P and is dropped; it also ranks after
// all of them, so leaving it out changes no mass-before of the others: the
// search runs over the keys at or above the highest threshold that holds P (at
// attention-like scores a few dozen, which the compare-count finishes without
// a histogram pass).  Sequences of more than 4096 blocks search all of their
// keys.
#include "../../include/up.h"
#include "common.cuh"

namespace up {

namespace {

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kBuckets = 4096;
constexpr int kSmallM = 64;  // keys left in the crossing bucket that a compare-count finishes
static_assert(16 * kSmallM == kSelThreads, "the compare-count gives each key 16 threads");
constexpr int kPasses = 5;

struct SelectShared {
    // bucket masses as two 32-bit words (native 32-bit shared atomics; the
    // carry out of the low word is added to the high word: exact)
    unsigned int mass_lo[kBuckets], mass_hi[kBuckets];
    unsigned int cnt[kBuckets];
    unsigned long long wsum[kSelWarps];
    unsigned long long mkey[kSmallM];
    unsigned long long mfx[kSmallM];
    unsigned long long base, kstar;
    int cross, m, nmem;
    int kept[kSelWarps];
    unsigned long long fmass[3][kSelWarps];  // threshold filter: per-warp masses and counts
    unsigned int fcnt[3][kSelWarps];
    unsigned int fT;                         // the filter's high-word bound (0xFFFFFFFF: none)
    int fM;                                  // keys it leaves
};

// High words of the filter's thresholds: score >= 2^-j <=> the rank key's high
// word (0x7FFFFFFF - score bits) <= 0x7FFFFFFF - ((127 - j) << 23).
__host__ __device__ constexpr unsigned filter_bound(int j) {
    return 0x7FFFFFFFu - ((unsigned)(127 - j) << 23);
}
constexpr int kFilters = 3;
__device__ __forceinline__ unsigned filter_threshold(int f) {
    return f == 0 ? filter_bound(8) : f == 1 ? filter_bound(14) : filter_bound(20);
}

__device__ __forceinline__ unsigned long long rank_key(float score, int idx) {
    // scores are >= 0; -0, NaN and anything not > 0 rank as 0.  The score bits
    // of a non-negative float fit in 31 bits, so the key's top bit is always 0
    // and its bits 62..55 are exactly the float's exponent.
    const unsigned bits = score > 0.f ? __float_as_uint(score) : 0u;
    return ((unsigned long long)(0x7FFFFFFFu - bits) << 32) | (unsigned)idx;
}

// score * 2^62 truncated, from the key's score bits; scores >= 1 count as 1.
__device__ __forceinline__ unsigned long long key_fixed(unsigned long long key) {
    const unsigned bits = 0x7FFFFFFFu - (unsigned)(key >> 32);
    if (bits >= 0x3F800000u) return 1ull << 62;
    const int e = (int)(bits >> 23);
    if (e == 0) return 0ull;  // zero or subnormal (< 2^-126)
    const unsigned long long m = (bits & 0x7FFFFFu) | 0x800000u;  // value = m * 2^(e-150)
    const int sh = e - 88;                                       // times 2^62
    return sh >= 0 ? (m << sh) : (sh > -24 ? (m >> -sh) : 0ull);
}

__device__ __forceinline__ void add_mass(SelectShared &sh, int b, unsigned long long v) {
    const unsigned lo = (unsigned)v;
    const unsigned old = atomicAdd(&sh.mass_lo[b], lo);
    atomicAdd(&sh.mass_hi[b], (unsigned)(v >> 32) + (old + lo < old ? 1u : 0u));
}

__device__ __forceinline__ unsigned long long bucket_mass(const SelectShared &sh, int b) {
    return ((unsigned long long)sh.mass_hi[b] << 32) | sh.mass_lo[b];
}

// digit of each pass: (shift, width); key bits 31..16 are always zero
__device__ __forceinline__ int pass_shift(int ps) {
    return ps == 0 ? 51 : ps == 1 ? 39 : ps == 2 ? 32 : ps == 3 ? 4 : 0;
}
__device__ __forceinline__ int pass_width(int ps) {
    return ps == 2 ? 7 : ps == 4 ? 4 : 12;
}

// CTA-wide exclusive scan of one u64 per thread; *total = the sum.
__device__ __forceinline__ unsigned long long block_scan_u64(unsigned long long v,
                                                             unsigned long long *total,
                                                             SelectShared &sh) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    unsigned long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh.wsum[wid] = x;
    __syncthreads();
    if (wid == 0) {
        unsigned long long w = lane < kSelWarps ? sh.wsum[lane] : 0ull;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kSelWarps) sh.wsum[lane] = w;
    }
    __syncthreads();
    *total = sh.wsum[kSelWarps - 1];
    return (wid ? sh.wsum[wid - 1] : 0ull) + x - v;
}

template <int E>
__device__ void select_seq(const float *__restrict__ scores, int b0, int nb, int L, int G,
                           unsigned long long P, bool unit_mass, bool keep_all, bool keep_last,
                           uint8_t *__restrict__ keep, int32_t *kept_tokens, int s,
                           SelectShared &sh) {
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    // the rank key's high word per key; its low word is the index t + i * kSelThreads
    unsigned khi[E];
#pragma unroll
    for (int i = 0; i < E; ++i) {
        const int e = t + i * kSelThreads;
        khi[i] = e < nb ? (unsigned)(rank_key(scores[b0 + e], e) >> 32) : 0u;
    }
    auto key = [&](int i) {
        return ((unsigned long long)khi[i] << 32) | (unsigned)(t + i * kSelThreads);
    };
    auto mass = [&](int i) { return unit_mass ? 1ull : key_fixed(key(i)); };
    unsigned long long kstar = ~0ull;  // keep-all
    if (!keep_all) {
        // the threshold filter: keys with a high word above T cannot be kept
        unsigned T = 0xFFFFFFFFu;
        int m = nb;
        if constexpr (E <= 4) {  // (longer sequences: registers are short, and they search all keys)
            unsigned long long fm[kFilters];
            unsigned fc[kFilters];
#pragma unroll
            for (int f = 0; f < kFilters; ++f) {
                fm[f] = 0ull;
                fc[f] = 0u;
            }
#pragma unroll
            for (int i = 0; i < E; ++i) {
                if (t + i * kSelThreads >= nb) continue;
                const unsigned long long mi = mass(i);
#pragma unroll
                for (int f = 0; f < kFilters; ++f)
                    if (khi[i] <= filter_threshold(f)) {
                        fm[f] += mi;
                        ++fc[f];
                    }
            }
#pragma unroll
            for (int f = 0; f < kFilters; ++f) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    fm[f] += __shfl_xor_sync(0xffffffffu, fm[f], o);
                    fc[f] += __shfl_xor_sync(0xffffffffu, fc[f], o);
                }
                if (lane == 0) {
                    sh.fmass[f][wid] = fm[f];
                    sh.fcnt[f][wid] = fc[f];
                }
            }
            __syncthreads();
            if (wid == 0) {
                unsigned bound = 0xFFFFFFFFu;
                int left = nb;
#pragma unroll
                for (int f = 0; f < kFilters; ++f) {
                    unsigned long long v = lane < kSelWarps ? sh.fmass[f][lane] : 0ull;
                    unsigned c = lane < kSelWarps ? sh.fcnt[f][lane] : 0u;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        v += __shfl_xor_sync(0xffffffffu, v, o);
                        c += __shfl_xor_sync(0xffffffffu, c, o);
                    }
                    if (bound == 0xFFFFFFFFu && v >= P) {  // the highest threshold that holds P
                        bound = filter_threshold(f);
                        left = (int)c;
                    }
                }
                if (lane == 0) {
                    sh.fT = bound;
                    sh.fM = left;
                }
            }
            __syncthreads();
            T = sh.fT;
            m = sh.fM;
        }
        unsigned long long prefix = 0ull, base = 0ull;
        int fixed_from = 64;  // key bits >= fixed_from are those of the crossing bucket
#pragma unroll 1
        for (int ps = 0; ps < kPasses && m > kSmallM; ++ps) {
            const int shift = pass_shift(ps), nbk = 1 << pass_width(ps);
            for (int b = t; b < nbk; b += kSelThreads) {
                sh.mass_lo[b] = 0u;
                sh.mass_hi[b] = 0u;
                sh.cnt[b] = 0u;
            }
            if (t == 0) sh.cross = -1;
            __syncthreads();
#pragma unroll
            for (int i = 0; i < E; ++i) {
                const int e = t + i * kSelThreads;
                const unsigned long long k = key(i);
                const bool member = e < nb && khi[i] <= T &&
                                    (fixed_from == 64 || (k >> fixed_from) == (prefix >> fixed_from));
                const int b = member ? (int)((k >> shift) & (unsigned long long)(nbk - 1)) : -1;
                const unsigned long long fx = member ? mass(i) : 0ull;
                // Neighbouring blocks often share a bucket (scores of similar
                // size), and atomics on one shared address serialise: a warp
                // first adds up, in up to four rounds, the masses of the lanes
                // that share its lowest pending lane's bucket (one atomic per
                // bucket and round); lanes still pending then add their own.
                unsigned pending = __ballot_sync(0xffffffffu, member);
#pragma unroll 1
                for (int round = 0; round < 4 && pending; ++round) {
                    const int leader = __ffs(pending) - 1;
                    const int d = __shfl_sync(0xffffffffu, b, leader);
                    const bool mine = member && b == d;
                    const unsigned peers = __ballot_sync(0xffffffffu, mine);
                    unsigned long long v = mine ? fx : 0ull;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (lane == leader) {
                        add_mass(sh, d, v);
                        atomicAdd(&sh.cnt[d], (unsigned)__popc(peers));
                    }
                    pending &= ~peers;
                }
                if ((pending >> lane) & 1u) {
                    add_mass(sh, b, fx);
                    atomicAdd(&sh.cnt[b], 1u);
                }
            }
            __syncthreads();
            // thread t owns buckets 4t .. 4t+3 (nbk <= 4096)
            const int per = (nbk + kSelThreads - 1) / kSelThreads;  // 1 or 4
            unsigned long long loc = 0ull;
            for (int j = 0; j < per; ++j) {
                const int b = t * per + j;
                if (b < nbk) loc += bucket_mass(sh, b);
            }
            unsigned long long tot;
            unsigned long long before = base + block_scan_u64(loc, &tot, sh);
            int best = -1;
            unsigned long long best_before = 0ull;
            for (int j = 0; j < per; ++j) {
                const int b = t * per + j;
                if (b < nbk) {
                    if (sh.cnt[b] > 0u && before < P) {
                        best = b;
                        best_before = before;
                    }
                    before += bucket_mass(sh, b);
                }
            }
            if (best >= 0) atomicMax(&sh.cross, best);
            __syncthreads();
            if (best >= 0 && best == sh.cross) {
                sh.base = best_before;
                sh.m = (int)sh.cnt[best];
            }
            __syncthreads();
            prefix |= (unsigned long long)sh.cross << shift;
            base = sh.base;
            m = sh.m;
            fixed_from = shift;
            __syncthreads();  // the next pass clears the buckets
        }
        // the keys of the crossing bucket (at most kSmallM): each takes its exact
        // mass-before by comparison; K* is the largest with mass-before < P
        if (t == 0) {
            sh.nmem = 0;
            sh.kstar = 0ull;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < E; ++i) {
            const int e = t + i * kSelThreads;
            const unsigned long long k = key(i);
            if (e < nb && khi[i] <= T &&
                (fixed_from == 64 || (k >> fixed_from) == (prefix >> fixed_from))) {
                const int slot = atomicAdd(&sh.nmem, 1);
                if (slot < kSmallM) {
                    sh.mkey[slot] = k;
                    sh.mfx[slot] = mass(i);
                }
            }
        }
        __syncthreads();
        const int nm = min(sh.nmem, kSmallM);
        {
            // 16 threads per key (kSelThreads = 16 * kSmallM), each summing the
            // masses of every 16th other key ranked before it
            const int mi = t >> 4, q = t & 15;
            const unsigned long long ki = mi < nm ? sh.mkey[mi] : 0ull;
            unsigned long long bf = 0ull;
            if (mi < nm)
                for (int j = q; j < nm; j += 16)
                    if (sh.mkey[j] < ki) bf += sh.mfx[j];
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) bf += __shfl_xor_sync(0xffffffffu, bf, o);
            if (mi < nm && q == 0 && base + bf < P) atomicMax(&sh.kstar, ki);
        }
        __syncthreads();
        kstar = sh.kstar;
    }
    int kept = 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
        const int e = t + i * kSelThreads;
        if (e < nb) {
            const int k = (key(i) <= kstar || (keep_last && e == nb - 1)) ? 1 : 0;
            keep[b0 + e] = (uint8_t)k;
            if (k) kept += min(G, L - e * G);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) kept += __shfl_xor_sync(0xffffffffu, kept, o);
    if (lane == 0) sh.kept[wid] = kept;
    __syncthreads();
    if (t < 32) {
        int w = t < kSelWarps ? sh.kept[t] : 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
        if (t == 0) kept_tokens[s] = w;
    }
}

// grid (num_seqs): one CTA per sequence.
__global__ void __launch_bounds__(kSelThreads, 1)
select_kernel(const float *__restrict__ scores, const int32_t *__restrict__ cu_blocks,
              const int32_t *__restrict__ cu, int G, unsigned long long P, int unit_mass,
              int keep_all, int keep_last, uint8_t *__restrict__ keep,
              int32_t *__restrict__ kept_tokens, unsigned int *err) {
    extern __shared__ __align__(16) unsigned char sel_smem[];
    SelectShared &sh = *reinterpret_cast<SelectShared *>(sel_smem);
    pdl_wait();
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
    // checked builds: this sequence's flags lie inside the batch's [0, cu_blocks[B])
    if (!in_range(b0, nb, cu_blocks[gridDim.x], err)) {
        if (threadIdx.x == 0) kept_tokens[s] = 0;
        return;
    }
    const bool all = keep_all != 0, unit = unit_mass != 0, last = keep_last != 0;
    if (nb <= kSelThreads) select_seq<1>(scores, b0, nb, L, G, P, unit, all, last, keep, kept_tokens, s, sh);
    else if (nb <= 2 * kSelThreads) select_seq<2>(scores, b0, nb, L, G, P, unit, all, last, keep, kept_tokens, s, sh);
    else if (nb <= 4 * kSelThreads) select_seq<4>(scores, b0, nb, L, G, P, unit, all, last, keep, kept_tokens, s, sh);
    else if (nb <= 8 * kSelThreads) select_seq<8>(scores, b0, nb, L, G, P, unit, all, last, keep, kept_tokens, s, sh);
    else select_seq<16>(scores, b0, nb, L, G, P, unit, all, last, keep, kept_tokens, s, sh);
}

}  // namespace

cudaError_t launch_select(const float *scores, const int32_t *cu_blocks, const int32_t *cu_seqlens,
                          int num_seqs, int G, bool top_k, double p, int k, bool keep_last,
                          uint8_t *keep, int32_t *kept_tokens, unsigned int *err, int num_sms,
                          cudaStream_t st) {
    (void)num_sms;
    if (num_seqs <= 0) return cudaSuccess;
    static_assert(UP_SELECT_MAX_BLOCKS <= 16 * kSelThreads, "select keeps at most 16 keys per thread");
    static_assert(UP_SELECT_MAX_BLOCKS <= 65536, "the index digits cover 16 bits");
    bool all;
    unsigned long long P;
    if (top_k) {
        all = k >= UP_SELECT_MAX_BLOCKS;  // every sequence that fits keeps everything
        P = (unsigned long long)k;
    } else {
        all = !(p < 1.0);
        // P = ceil(p * 2^62): p * 2^62 is exact in fp64, so this is the exact threshold
        P = all ? 0ull : (unsigned long long)ceil(p * 4611686018427387904.0);
    }
    const int smem = (int)sizeof(SelectShared);
    const cudaError_t attr =
        cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (attr != cudaSuccess) return attr;
    if (num_seqs > 2147483647) return cudaErrorInvalidValue;
    return launch_pdl(select_kernel, dim3(num_seqs), dim3(kSelThreads), (size_t)smem, st, scores,
                      cu_blocks, cu_seqlens, G, P, top_k ? 1 : 0, all ? 1 : 0, keep_last ? 1 : 0,
                      keep, kept_tokens, err);
}

}  // namespace up
