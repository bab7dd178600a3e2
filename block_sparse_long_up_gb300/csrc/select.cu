// select.cu -- top-p block selection, one CTA per sequence.
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
// mass-before is < P (top-p: P = ceil(p * 2^62)).  K* is found by a radix search over the
// key's digits, most significant first.  Each pass histograms the exact masses
// (and counts) of the keys that share the digits found so far over the next
// 8-bit digit (a warp first adds the masses of its lanes that share a digit,
// so the shared-memory atomics stay few even when the leading digits barely
// vary); the last non-empty bucket whose mass-before is < P holds K*
// (the first key of that bucket is kept; the first key of any later bucket is
// not).  A bucket holding a single key ends the search.  Six passes at most:
// four over the 31 score bits (the first is the exponent), two over the block
// index (< 2^16).
//
// A single sequence of at most kCmpMaxBlocks blocks skips the search: about
// two CTAs per SM share it, each loads all of its keys into shared memory, and
// one warp per block takes the exact mass-before of the block directly, as the
// sum of the masses of every key ranked before it (nb^2 key comparisons, spread
// over the GPU).  The same rule decides: kept iff mass-before < P.  The block at
// the last kept rank (mass-before < P and, with its own mass, >= P, or no key
// ranked after it) writes the sequence's kept tokens, so no CTA waits for
// another.  Several sequences take the search, one CTA each, side by side (an
// even split of the CTAs over sequences of unequal length measured slower).
#include <algorithm>

#include "../../include/up.h"
#include "common.cuh"

namespace up {

namespace {

constexpr int kSelThreads = 512;
constexpr int kCmpMaxBlocks = 4096;  // larger sequences take the radix search
constexpr int kCmpSmem = 2 * kCmpMaxBlocks * (int)sizeof(unsigned long long);

__device__ __forceinline__ unsigned long long rank_key(float score, int idx) {
    // scores are >= 0; -0, NaN and anything not > 0 rank as 0.  The score bits
    // of a non-negative float fit in 31 bits, so the key's top bit is always 0
    // and its first radix digit (bits 55..62) is exactly the float's exponent.
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

// Shared state of one selection.  Bucket masses are kept as four 16-bit
// pieces (each sum < 2^30 for <= 2^14 keys) plus counts.
struct SelectShared {
    alignas(16) unsigned int hpart[4][256];
    alignas(16) unsigned int hcnt[256];
    unsigned long long s_prefix, s_base, s_kstar;
    unsigned int s_cnt;
    int shi[32];
};

template <int E>
__device__ void select_one(const float *__restrict__ scores, int b0, int nb, int L, int G,
                           unsigned long long P, bool unit_mass, bool keep_all, bool keep_last,
                           uint8_t *__restrict__ keep, int32_t *kept_tokens, int s,
                           SelectShared &sh) {
    auto &hpart = sh.hpart;
    auto &hcnt = sh.hcnt;
    auto &s_prefix = sh.s_prefix;
    auto &s_base = sh.s_base;
    auto &s_kstar = sh.s_kstar;
    auto &s_cnt = sh.s_cnt;
    auto &shi = sh.shi;
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
    unsigned long long kstar = ~0ull;  // keep-all
    if (!keep_all) {
        unsigned long long prefix = 0ull, base = 0ull;
        bool single = false;
#pragma unroll 1
        for (int ps = 0; ps < 6; ++ps) {
            // digits: exponent (55..62), mantissa 47..54, 39..46, 32..39 (bit 39 is
            // already fixed by then), then the block index (16 bits)
            const int sh = ps < 3 ? 55 - 8 * ps : (ps == 3 ? 32 : 40 - 8 * ps);  // 55,47,39,32,8,0
            if (t < 256) {
#pragma unroll
                for (int k = 0; k < 4; ++k) hpart[k][t] = 0u;
                hcnt[t] = 0u;
            }
            __syncthreads();
#pragma unroll
            for (int i = 0; i < E; ++i) {
                const int e = t + i * kSelThreads;
                const bool match = ps == 0 || (key(i) >> (sh + 8)) == (prefix >> (sh + 8));
                // 256 = not in the searched range.  A warp aggregates by digit:
                // in up to four rounds it takes the digit of its lowest pending
                // lane, adds the masses of all lanes holding that digit with a
                // shuffle tree, and one lane updates the bucket; lanes still
                // pending after that update their own buckets.  The leading
                // digits take few distinct values per warp, so few atomics hit
                // the shared histogram.
                const unsigned dgt = (e < nb && match) ? (unsigned)((key(i) >> sh) & 255u) : 256u;
                const unsigned long long fx =
                    dgt < 256u ? (unit_mass ? 1ull : key_fixed(key(i))) : 0ull;
                unsigned pending = __ballot_sync(0xffffffffu, dgt < 256u);
#pragma unroll 1
                for (int round = 0; round < 4 && pending; ++round) {
                    const int leader = __ffs(pending) - 1;
                    const unsigned d = __shfl_sync(0xffffffffu, dgt, leader);
                    const bool mine = dgt == d;
                    const unsigned peers = __ballot_sync(0xffffffffu, mine);
                    unsigned long long v = mine ? fx : 0ull;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (lane == leader) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            atomicAdd(&hpart[k][d], (unsigned)(v >> (16 * k)) & 0xFFFFu);
                        atomicAdd(&hcnt[d], (unsigned)__popc(peers));
                    }
                    pending &= ~peers;
                }
                if ((pending >> lane) & 1u) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        atomicAdd(&hpart[k][dgt], (unsigned)(fx >> (16 * k)) & 0xFFFFu);
                    atomicAdd(&hcnt[dgt], 1u);
                }
            }
            __syncthreads();
            if (wid == 0) {
                // lane l owns buckets 8l .. 8l+7 (read as 16-byte vectors):
                // exclusive scan of the lane totals
                unsigned pc[4][8], cc[8];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint4 a = reinterpret_cast<const uint4 *>(&hpart[k][8 * lane])[0];
                    const uint4 b = reinterpret_cast<const uint4 *>(&hpart[k][8 * lane])[1];
                    pc[k][0] = a.x; pc[k][1] = a.y; pc[k][2] = a.z; pc[k][3] = a.w;
                    pc[k][4] = b.x; pc[k][5] = b.y; pc[k][6] = b.z; pc[k][7] = b.w;
                }
                {
                    const uint4 a = reinterpret_cast<const uint4 *>(&hcnt[8 * lane])[0];
                    const uint4 b = reinterpret_cast<const uint4 *>(&hcnt[8 * lane])[1];
                    cc[0] = a.x; cc[1] = a.y; cc[2] = a.z; cc[3] = a.w;
                    cc[4] = b.x; cc[5] = b.y; cc[6] = b.z; cc[7] = b.w;
                }
                auto bucket_mass = [&](int j) {
                    return (unsigned long long)pc[0][j] + ((unsigned long long)pc[1][j] << 16) +
                           ((unsigned long long)pc[2][j] << 32) + ((unsigned long long)pc[3][j] << 48);
                };
                unsigned long long tot = 0ull;
#pragma unroll
                for (int j = 0; j < 8; ++j) tot += bucket_mass(j);
                unsigned long long x = tot;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
                    if (lane >= o) x += y;
                }
                unsigned long long S = base + (x - tot);  // mass before the lane's first bucket
                int best = -1;
                unsigned long long best_S = 0ull;
                unsigned best_c = 0u;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (cc[j] > 0u && S < P) {
                        best = 8 * lane + j;
                        best_S = S;
                        best_c = cc[j];
                    }
                    S += bucket_mass(j);
                }
                int top = best;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) top = max(top, __shfl_xor_sync(0xffffffffu, top, o));
                if (best == top && best >= 0) {
                    s_prefix = prefix | ((unsigned long long)best << sh);
                    s_base = best_S;
                    s_cnt = best_c;
                }
            }
            __syncthreads();
            prefix = s_prefix;
            base = s_base;
            if (s_cnt == 1u) {  // the bucket's only key is K*
#pragma unroll
                for (int i = 0; i < E; ++i) {
                    const int e = t + i * kSelThreads;
                    if (e < nb && (key(i) >> sh) == (prefix >> sh)) s_kstar = key(i);
                }
                single = true;
            }
            __syncthreads();
            if (single) break;
        }
        kstar = single ? s_kstar : prefix;
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
    if (lane == 0) shi[wid] = kept;
    __syncthreads();
    if (t < 32) {
        int w = t < kSelThreads / 32 ? shi[t] : 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
        if (t == 0) kept_tokens[s] = w;
    }
}

// Blocks [x * per, (x + 1) * per) of the sequence, per = ceil(nb / X).
__device__ void select_compare(const float *__restrict__ scores, int b0, int nb, int L, int G,
                               unsigned long long P, bool unit_mass, bool keep_all,
                               bool keep_last, uint8_t *__restrict__ keep,
                               int32_t *kept_tokens, int s, int x, int X,
                               unsigned long long *smem) {
    const int per = (nb + X - 1) / X;
    const int lo = x * per, hi = min(lo + per, nb);
    if (lo >= hi) return;
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    if (keep_all) {
        for (int e = lo + t; e < hi; e += kSelThreads) keep[b0 + e] = 1;
        if (x == 0 && t == 0) kept_tokens[s] = L;
        return;
    }
    unsigned long long *skey = smem, *sfx = smem + kCmpMaxBlocks;
#pragma unroll 4
    for (int e = t; e < nb; e += kSelThreads) {
        const unsigned long long k = rank_key(scores[b0 + e], e);
        skey[e] = k;
        sfx[e] = unit_mass ? 1ull : key_fixed(k);
    }
    __syncthreads();
    for (int i = lo + wid; i < hi; i += kSelThreads / 32) {
        const unsigned long long ki = skey[i];
        unsigned long long before = 0ull;
        bool after = false;  // some key ranks after block i
#pragma unroll 4
        for (int j = lane; j < nb; j += 32) {
            const unsigned long long kj = skey[j];
            if (kj < ki) before += sfx[j];
            after |= kj > ki;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
        after = __any_sync(0xffffffffu, after);
        const bool in = before < P;
        if (lane == 0) keep[b0 + i] = (in || (keep_last && i == nb - 1)) ? 1 : 0;
        if (in && (!after || before + sfx[i] >= P)) {  // the last kept rank
            int tok = 0;
            for (int j = lane; j < nb; j += 32)
                if (skey[j] <= ki || (keep_last && j == nb - 1)) tok += min(G, L - j * G);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) tok += __shfl_xor_sync(0xffffffffu, tok, o);
            if (lane == 0) kept_tokens[s] = tok;
        }
    }
}

// grid (X, num_seqs): CTA x of sequence blockIdx.y (X > 1 only for one sequence).
__global__ void __launch_bounds__(kSelThreads, 2)
select_topp_kernel(const float *__restrict__ scores, const int32_t *__restrict__ cu_blocks,
                   const int32_t *__restrict__ cu, int G, unsigned long long P, int unit_mass,
                   int keep_all, int keep_last, uint8_t *__restrict__ keep,
                   int32_t *__restrict__ kept_tokens, unsigned int *err) {
    extern __shared__ __align__(16) unsigned long long cmp_smem[];
    pdl_wait();
    const int s = blockIdx.y, x = blockIdx.x;
    const int b0 = cu_blocks[s];
    const int nb = cu_blocks[s + 1] - b0;
    const int L = cu[s + 1] - cu[s];
    if (nb <= 0) {
        if (x == 0 && threadIdx.x == 0) kept_tokens[s] = 0;
        return;
    }
    if (nb > UP_SELECT_MAX_BLOCKS) {
        if (x == 0 && threadIdx.x == 0) {
            atomicOr(err, UP_DEVERR_SELECT_TOO_MANY_BLOCKS);
            kept_tokens[s] = 0;
        }
        return;
    }
    const bool all = keep_all != 0, unit = unit_mass != 0, last = keep_last != 0;
    if (gridDim.x > 1 && nb <= kCmpMaxBlocks) {
        select_compare(scores, b0, nb, L, G, P, unit, all, last, keep, kept_tokens, s, x,
                       (int)gridDim.x, cmp_smem);
        return;
    }
    if (x != 0) return;
    __shared__ SelectShared sh;
    if (nb <= kSelThreads) select_one<1>(scores, b0, nb, L, G, P, unit, all, last, keep, kept_tokens, s, sh);
    else if (nb <= 2 * kSelThreads) select_one<2>(scores, b0, nb, L, G, P, unit, all, last, keep, kept_tokens, s, sh);
    else if (nb <= 4 * kSelThreads) select_one<4>(scores, b0, nb, L, G, P, unit, all, last, keep, kept_tokens, s, sh);
    else if (nb <= 8 * kSelThreads) select_one<8>(scores, b0, nb, L, G, P, unit, all, last, keep, kept_tokens, s, sh);
    else if (nb <= 16 * kSelThreads) select_one<16>(scores, b0, nb, L, G, P, unit, all, last, keep, kept_tokens, s, sh);
    else select_one<32>(scores, b0, nb, L, G, P, unit, all, last, keep, kept_tokens, s, sh);
}

}  // namespace

cudaError_t launch_select(const float *scores, const int32_t *cu_blocks, const int32_t *cu_seqlens,
                          int num_seqs, int G, bool top_k, double p, int k, bool keep_last,
                          uint8_t *keep, int32_t *kept_tokens, unsigned int *err, int num_sms,
                          cudaStream_t st) {
    if (num_seqs <= 0) return cudaSuccess;
    static_assert(UP_SELECT_MAX_BLOCKS <= 32 * kSelThreads, "select keeps at most 32 keys per thread");
    static_assert(UP_SELECT_MAX_BLOCKS <= 65536, "the radix search covers 16 index bits");
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
    const cudaError_t attr = cudaFuncSetAttribute(
        select_topp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kCmpSmem);
    if (attr != cudaSuccess) return attr;
    // one sequence: about two CTAs per SM share it; several: one CTA each
    const int X = num_seqs == 1 ? std::max(2, 2 * num_sms) : 1;
    if (num_seqs > 65535) return cudaErrorInvalidValue;
    return launch_pdl(select_topp_kernel, dim3(X, num_seqs), dim3(kSelThreads),
                      X > 1 ? (size_t)kCmpSmem : 0, st, scores, cu_blocks, cu_seqlens, G, P,
                      top_k ? 1 : 0, all ? 1 : 0, keep_last ? 1 : 0, keep, kept_tokens, err);
}

}  // namespace up
