// score_tc.cu -- block scoring on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// UniPrefill overview, block-wise importance estimation paragraph: the last n
// queries of a sequence are dotted with all of its keys, the softmax mass of
// each query is summed over fixed blocks of G keys and averaged over queries
// and heads.  Its fused-kernel paragraph names the pieces fused here: loads from
// HBM, online softmax and block reduction in one pipeline.
//
// Work unit = (sequence s, KV head j, group of 128-row tiles, key chunk c).  The
// rows are the packed GQA rows of KV head j (query t of head j*g + h is row
// t*g + h), so one K step serves every query head that shares it (the PackGQA
// idea of the FlashPrefill V2 review, re-derived for tcgen05).  A unit holds
// four row tiles (512 rows: all query heads of a KV head at n = 128) when
// head_dim <= 128, so each K byte enters shared memory once.  Tiles are handled
// in pairs; the two TMEM buffers (2 tiles x 128 fp32 columns each) alternate
// between pairs (head_dim <= 128: pair p always uses buffer p) or between K
// steps (head_dim 256: one pair per unit).
// A persistent CTA per SM walks its units; roles are warp-specialised:
//   warp 0      K producer: TMA loads of 128-key x 64-dim K panels (128-byte
//               swizzle) into a ring of shared-memory stages (keys token-major,
//               or through a block table from a paged KV-head-major cache);
//   warp 2      Q producer: TMA loads of each pair's Q tiles (one 3-D box of
//               g heads x 128/g queries x 64 dims per tile and panel);
//   warps 1, 3  MMA issuers, one per TMEM buffer: S = Q K^T as M=128, N=128
//               tcgen05.mma chains, each K slice issued to the pair's two
//               tiles in turn (consecutive MMAs never share an accumulator).
//               The whole warp walks the loop and one elected lane issues, so
//               the bookkeeping of one issuer (barrier waits, commits) runs
//               while the other one's MMAs keep the pipe busy (head_dim 256:
//               each K panel is multiplied and released as soon as it lands);
//   warps 4-11  two softmax warpgroups; warpgroup e owns tile e of each pair.
//               Thread = row (TMEM lane).  It reads 32 columns at a time (the
//               next group's TMEM load in flight while the current one is
//               processed), applies the causal mask on the last steps, computes
//               2^(z*log2e/sqrt(d) - ref) on the MUFU and sums each block of G
//               keys; the block sums go straight to HBM as partials.
// The reference `ref` of a row is the largest visible logit among the first 32
// keys of the unit; the row's statistics for the chunk (ref and the sum of all
// its block partials) go to workspace.  Later keys may exceed ref; fp32 absorbs
// that up to ~115 binary orders of magnitude, and a tile whose sums overflow
// anyway is queued for an exact CUDA-core fallback in the epilogue.  After its
// last unit every CTA runs the epilogue: grid barriers, then each row's
// normaliser and chunk weights, then the block scores (see score_epilogue).
#include <cudaTypedefs.h>

#include "../../include/up.h"
#include "common.cuh"
#include "sm100.cuh"

namespace up {

namespace {

using namespace sm100;

constexpr int kWarpTmaK = 0;
constexpr int kWarpMma0 = 1;     // issues the MMAs of TMEM buffer 0
constexpr int kWarpTmaQ = 2;
constexpr int kWarpMma1 = 3;     // issues the MMAs of TMEM buffer 1
constexpr int kWarpEpi = 4;      // warps 4..11: two warpgroups
constexpr int kEpiThreads = 128; // one warpgroup
constexpr int kPanelBytesK = kStepKeys * 128;      // 128 keys x 64 bf16 = 16 KB
constexpr int kPanelBytesQ = kRowsPerTile * 128;   // 128 rows x 64 bf16 = 16 KB
constexpr uint32_t kTmemCols = 512;
constexpr int kBufCols = 2 * kStepKeys;            // one TMEM buffer: a pair of tiles
constexpr int kSmemBudget = 227 * 1024 - 2048;     // dynamic bytes we allow ourselves
constexpr long long kWaitLimit = 4000000000LL;     // cycles, ~2 s: the drain after an abort
constexpr int kMaxStages = 16;

template <int D>
struct Cfg {
    // Two softmax warpgroups (warpgroup e takes tile e of every pair).  Four
    // (one tile each at head_dim <= 128) measured slower: only two TMEM buffers
    // of two tiles fit, so the warpgroups of a buffer idle while it is refilled.
    static constexpr int kWGs = 2;
    static constexpr int kThreads = 128 * (1 + kWGs);
    static constexpr int kTiles = tiles_per_unit(D);
    static constexpr int kPairs = kTiles / 2;
    static constexpr int kPanels = D / 64;
    static constexpr int kQTileBytes = kPanels * kPanelBytesQ;   // one row tile
    static constexpr int kQPairBytes = 2 * kQTileBytes;          // the Q tiles of one pair
    static constexpr int kQBytes = kTiles * kQTileBytes;         // one Q buffer (all pairs)
    static constexpr int kQBufs = (2 * kQBytes + 6 * kPanelBytesK <= kSmemBudget) ? 2 : 1;
    static constexpr int kQSlots = kQBufs * kPairs;              // pair buffers
    static constexpr int kStagesFit = (kSmemBudget - 1024 - kQBufs * kQBytes) / kPanelBytesK;
    static constexpr int kStages = kStagesFit < kMaxStages ? kStagesFit : kMaxStages;
    static constexpr int kSmem = kQBufs * kQBytes + kStages * kPanelBytesK + 1024;
    // both issuers read every K stage and every Q pair buffer (one tile each)
    static constexpr int kStageUsers = 2;
    static constexpr int kQUsers = 2;
    static_assert(kStages >= kPanels, "at least one K step in flight");
    static_assert(kTiles % 2 == 0 && kPairs <= 2, "tile pairs map onto the two TMEM buffers");
    static_assert(kQSlots <= 4, "Q pair buffers");
};

struct Shared {
    uint64_t kfull[kMaxStages], kempty[kMaxStages];
    uint64_t qfull[4], qempty[4];  // one per pair buffer
    uint64_t tfull[2], tempty[2];
    uint64_t fin[2];
    uint32_t tmem_base;
    int units;
    int abort;
    int epi_state;  // epilogue: 0 go on, 1 a wait expired, 2 tiles were queued for the exact fallback
};

struct Unit {
    SeqInfo sq;
    int s;  // sequence index
    int j, grp, c, k0, k1, nsteps;
    int npairs;  // pairs of row tiles holding at least one query (a prefix of the pairs)
};

template <int D>
__device__ __forceinline__ void decode_unit(const ScoreParams &p, int u, Unit &un) {
    using C = Cfg<D>;
    if (p.num_seqs == 1) {
        un.s = 0;
        un.sq = p.seq0;
    } else {
        un.s = find_seq_by_unit(p.seqs, p.num_seqs, u);
        un.sq = p.seqs[un.s];
    }
    int loc = u - un.sq.unit_off;
    un.grp = loc % un.sq.mtiles;  // group of row tiles
    loc /= un.sq.mtiles;
    un.c = loc % un.sq.nchunks;
    un.j = loc / un.sq.nchunks;
    un.k0 = un.c * p.C;
    un.k1 = min(un.k0 + p.C, un.sq.L);
    un.nsteps = (un.k1 - un.k0 + kStepKeys - 1) / kStepKeys;
    const int left = un.sq.ns - un.grp * C::kTiles * p.tpt;  // > 0: the group holds queries
    un.npairs = min(C::kPairs, (left + 2 * p.tpt - 1) / (2 * p.tpt));
}

// The query (relative to the sequence) a row tile's tensor-map box starts at.
// A tile's own queries start at tile * tpt; the last tile of a sequence is
// shifted back so that its box ends at the sequence's last query and never
// reads past q_last (whose length only the device knows).  The shifted box's
// leading rows repeat queries of the previous tile and count as unused.
__device__ __forceinline__ int tile_box_query(const ScoreParams &p, int ns, int tile) {
    return min(tile * p.tpt, ns - p.tpt);
}

// Waits for an operation already issued to finish, without looking at the
// abort flag (used when shutting down after an abort).
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kWaitLimit) break;
    }
}

// ---------------------------------------------------------------- roles

template <int D>
__device__ void role_tma_k(const CUtensorMap *tmap, const ScoreParams &p, Shared &sh,
                           uint8_t *kbuf, int units) {
    using C = Cfg<D>;
    volatile int *abort = &sh.abort;
    // K is read exactly once: its lines should leave L2 before the block
    // partials, which the epilogue reads back
    const uint64_t policy = l2_policy_evict_first();
    uint32_t it = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        Unit un;
        decode_unit<D>(p, u, un);
        for (int t = 0; t < un.nsteps; ++t) {
            // the step's 128 keys: rows of k as [tokens, Hk*d] (x = head's dims),
            // or of the paged keys as [pages*Hk*page_size, d] (a step never
            // straddles two pages)
            const int tok = un.k0 + t * kStepKeys;
            int x0 = un.j * D, row0 = un.sq.tok_off + tok;
            if (p.block_table) {
                x0 = 0;
                row0 = (int)paged_row(p, un.s, un.j, tok);
            }
            for (int pn = 0; pn < C::kPanels; ++pn, ++it) {
                const int st = it % C::kStages;
                const uint32_t ph = (it / C::kStages) & 1;
                if (!mbar_wait(smem_u32(&sh.kempty[st]), ph ^ 1, abort, p.wait_limit)) goto done;
                mbar_arrive_expect_tx(smem_u32(&sh.kfull[st]), kPanelBytesK);
                tma_load_2d_hint(smem_u32(kbuf + st * kPanelBytesK), tmap, x0 + pn * 64, row0,
                                 smem_u32(&sh.kfull[st]), policy);
            }
        }
    }
done:
    if (!*abort) return;
    // after an abort nobody consumes the loads already issued: let them land
    // before the CTA can exit
    for (uint32_t k = 0; k < (uint32_t)C::kStages && k < it; ++k) {
        const uint32_t i = it - 1 - k;
        mbar_drain(smem_u32(&sh.kfull[i % C::kStages]), (i / C::kStages) & 1);
    }
}

// Q producer: for each unit and each pair of its row tiles that holds queries,
// waits for the pair's buffer and loads both tiles with one 3-D box per tile and
// 64-dim panel: {64 dims, g heads, tpt queries} of q_last viewed as
// [queries][Hq][d], which lands as 128-byte rows (row = query * g + head) in the
// K-major 128-byte-swizzled layout the MMA reads.
template <int D>
__device__ void role_tma_q(const CUtensorMap *tmap, const ScoreParams &p, Shared &sh,
                           uint8_t *qbuf, int units) {
    using C = Cfg<D>;
    volatile int *abort = &sh.abort;
    const uint32_t tx = (uint32_t)(2 * C::kPanels * 128 * p.g * p.tpt);
    // per pair buffer qs: bit qs of `parity` = parity of the loads issued into it
    // so far, bit qs of `used` = at least one load issued
    uint32_t parity = 0u, used = 0u;
    uint32_t ui = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++ui) {
        Unit un;
        decode_unit<D>(p, u, un);
        for (int pr = 0; pr < un.npairs; ++pr) {
            const int qs = (ui % C::kQBufs) * C::kPairs + pr;
            if (!mbar_wait(smem_u32(&sh.qempty[qs]), ((parity >> qs) & 1u) ^ 1u, abort, p.wait_limit))
                goto done;
            mbar_arrive_expect_tx(smem_u32(&sh.qfull[qs]), tx);
            for (int e = 0; e < 2; ++e) {
                const int tile = un.grp * C::kTiles + 2 * pr + e;
                const int z = un.sq.q_off + tile_box_query(p, un.sq.ns, tile);
                for (int pn = 0; pn < C::kPanels; ++pn)
                    tma_load_3d(smem_u32(qbuf + qs * C::kQPairBytes + e * C::kQTileBytes +
                                         pn * kPanelBytesQ),
                                tmap, pn * 64, un.j * p.g, z, smem_u32(&sh.qfull[qs]));
            }
            parity ^= 1u << qs;
            used |= 1u << qs;
        }
    }
done:
    if (!*abort) return;
    // the latest load into each used buffer completes phase parity ^ 1
    for (int qs = 0; qs < C::kQSlots; ++qs)
        if ((used >> qs) & 1u) mbar_drain(smem_u32(&sh.qfull[qs]), ((parity >> qs) & 1u) ^ 1u);
}

// MMA issuer w (0 or 1) issues the MMAs of tile w of every pair, so both
// issuers fill each TMEM buffer together, one accumulator each.  Slot order
// (the softmax warpgroups follow the same one): for each unit, each K step,
// each pair holding queries; head_dim <= 128: pair p uses buffer p; head_dim
// 256 (one pair): buffer = parity of the CTA-wide K step count.  Both issuers
// walk every K stage and Q pair buffer and release each after their last MMA
// on it, and each commits once to the buffer's full barrier.
// Two instruction streams keep the tensor pipe fed while the softmax warps
// load their sub-partitions' issue slots: one issuer alternating two
// accumulators got one M128 x N128 MMA per ~104 cycles under the softmax's
// load, two issuers ~65 (the full rate).  The whole warp walks the loop
// (warp-uniform control flow and descriptors) and one elected lane issues.
template <int D>
__device__ void role_mma(const ScoreParams &p, Shared &sh, uint8_t *qbuf, uint8_t *kbuf,
                         uint32_t tmem, int units, int w) {
    using C = Cfg<D>;
    constexpr uint32_t idesc = idesc_bf16_f32(kRowsPerTile, kStepKeys);
    volatile int *abort = &sh.abort;
    const bool leader = elect_one();
    uint32_t it = 0, gstep = 0;
    uint32_t tuse = 0u;  // bit b: parity of this issuer's uses of TMEM buffer b so far
    uint32_t qpar = 0u;  // bit qs: parity of the Q loads into pair buffer qs so far
    const uint32_t kbase = smem_u32(kbuf), qbase = smem_u32(qbuf);
    uint32_t ui = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++ui) {
        Unit un;
        decode_unit<D>(p, u, un);
        const int qb = (ui % C::kQBufs) * C::kPairs;
        uint32_t q_ready = 0u;  // bit pr: pair pr's Q seen loaded
        for (int t = 0; t < un.nsteps; ++t, ++gstep) {
            const uint32_t it0 = it;
            it += C::kPanels;
            if constexpr (C::kPairs == 2) {
                // head_dim <= 128: every K panel of the step is in shared memory
                // before the first MMA; the stage releases come after the last
                for (int pn = 0; pn < C::kPanels; ++pn) {
                    const uint32_t i = it0 + pn;
                    if (!mbar_wait_warp(smem_u32(&sh.kfull[i % C::kStages]), (i / C::kStages) & 1,
                                        abort, p.wait_limit))
                        goto out;
                }
            }
            for (int pr = 0; pr < C::kPairs; ++pr) {
                if (pr >= un.npairs) break;
                const int qs = qb + pr;
                const int buf = C::kPairs == 2 ? pr : (int)(gstep & 1u);
                if (!((q_ready >> pr) & 1u)) {
                    if (!mbar_wait_warp(smem_u32(&sh.qfull[qs]), (qpar >> qs) & 1u, abort,
                                        p.wait_limit))
                        goto out;
                    q_ready |= 1u << pr;
                }
                if (!mbar_wait_warp(smem_u32(&sh.tempty[buf]), ((tuse >> buf) & 1u) ^ 1u, abort,
                                    p.wait_limit))
                    goto out;
                tuse ^= 1u << buf;
                tc_fence_after();
                const uint32_t d_tile = tmem + (uint32_t)(buf * kBufCols + w * kStepKeys);
                const uint32_t qt = qbase + qs * C::kQPairBytes + w * C::kQTileBytes;
#pragma unroll 1
                for (int pn = 0; pn < C::kPanels; ++pn) {
                    const uint32_t i = it0 + pn;
                    const uint32_t st = i % C::kStages;
                    if constexpr (C::kPairs == 1) {
                        // head_dim 256: each panel is multiplied as soon as it
                        // lands and released right after (the ring holds six
                        // panels of a four-panel step)
                        if (!mbar_wait_warp(smem_u32(&sh.kfull[st]), (i / C::kStages) & 1, abort,
                                            p.wait_limit))
                            goto out;
                        tc_fence_after();
                    }
                    const uint64_t bd = smem_desc_sw128(kbase + st * kPanelBytesK);
                    const uint64_t ad = smem_desc_sw128(qt + pn * kPanelBytesQ);
                    if (leader) {
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)  // 4 x K=16 per 64-wide panel (32 B)
                            mma_bf16(d_tile, ad + 2 * ks, bd + 2 * ks, idesc, (pn | ks) != 0);
                        if constexpr (C::kPairs == 1) mma_commit(smem_u32(&sh.kempty[st]));
                    }
                    __syncwarp();
                }
                if (leader) mma_commit(smem_u32(&sh.tfull[buf]));
                __syncwarp();
            }
            if constexpr (C::kPairs == 1) {
                // a step without the pair (no queries) still releases its panels
                if (un.npairs == 0) {
                    for (int pn = 0; pn < C::kPanels; ++pn) {
                        const uint32_t i = it0 + pn;
                        if (!mbar_wait_warp(smem_u32(&sh.kfull[i % C::kStages]),
                                            (i / C::kStages) & 1, abort, p.wait_limit))
                            goto out;
                        if (leader) mma_commit(smem_u32(&sh.kempty[i % C::kStages]));
                        __syncwarp();
                    }
                }
            } else {
                if (leader) {
                    for (int pn = 0; pn < C::kPanels; ++pn)
                        mma_commit(smem_u32(&sh.kempty[(it0 + pn) % C::kStages]));
                }
                __syncwarp();
            }
        }
        // each pair buffer is free once this issuer's MMAs on it have completed
        for (int pr = 0; pr < un.npairs; ++pr) {
            if (leader) mma_commit(smem_u32(&sh.qempty[qb + pr]));
            __syncwarp();
            qpar ^= 1u << (qb + pr);
        }
    }
out:
    // every MMA issued by this warp has completed once fin fires
    if (leader) mma_commit(smem_u32(&sh.fin[w]));
    __syncwarp();
    mbar_drain(smem_u32(&sh.fin[w]), 0);
}

// One 32-column group: scale, shift, exponentiate, and return the sums of
// columns 0..15 (lo) and 16..31 (hi).  The scale and shift use packed fp32 FMAs
// on adjacent columns (which TMEM loads deliver in register pairs), the
// exponentials run on the MUFU, and the sums are a fixed tree of packed adds
// (even and odd columns apart until the last add): bitwise reproducible.
__device__ __forceinline__ void exp_sums(float (&v)[32], uint64_t s2, uint64_t bias2, float &lo,
                                         float &hi) {
    uint64_t e[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float z0, z1;
        unpack2(fma2(pack2(v[2 * i], v[2 * i + 1]), s2, bias2), z0, z1);
        e[i] = pack2(ex2_approx(z0), ex2_approx(z1));
    }
    const uint64_t l = add2(add2(add2(e[0], e[1]), add2(e[2], e[3])),
                            add2(add2(e[4], e[5]), add2(e[6], e[7])));
    const uint64_t h = add2(add2(add2(e[8], e[9]), add2(e[10], e[11])),
                            add2(add2(e[12], e[13]), add2(e[14], e[15])));
    float x, y;
    unpack2(l, x, y);
    lo = x + y;
    unpack2(h, x, y);
    hi = x + y;
}

// Causal mask of one group: keys past the row's limit a contribute nothing.
__device__ __forceinline__ void mask_group(float (&v)[32], int key, int a) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = (key + i > a) ? -INFINITY : v[i];
}

// One predicated store (no branch, so the group code stays one basic block),
// with an L2 evict-last policy: the epilogue reads the partials back.
__device__ __forceinline__ void st_if(float *p, float v, bool ok, uint64_t policy) {
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t"
        "@q st.global.L2::cache_hint.f32 [%0], %1, %3;\n\t}" ::"l"(p),
        "f"(v), "r"((int)ok), "l"(policy)
        : "memory");
}

// Per-row state of one row tile within a unit.
struct RowState {
    float *part;  // partial sums of this row: part[b * R]
    uint64_t policy;  // L2 policy of the partial stores
    float ref, lsum, acc;
    uint64_t bias2;
    int a;        // causal limit (absolute key position)
    int64_t r;    // row within the sequence
    bool valid;
};

// A K step of one row tile, general case: the unit's first step (which sets
// the reference) and the steps that reach the causal limit or the end of the
// sequence (masked, and their blocks may run past the sequence's last one).
template <int G>
__device__ __forceinline__ void softmax_tile(const Unit &un, RowState &rs, uint32_t taddr, int t,
                                             uint64_t s2, float s, Shared &sh, int buf) {
    constexpr int kGroups = kStepKeys / 32;
    constexpr int kGroupsPerBlock = G >= 32 ? G / 32 : 1;
    const SeqInfo &sq = un.sq;
    const int skey = un.k0 + t * kStepKeys;  // first key of the step
    const bool masked = skey + kStepKeys - 1 > sq.L - sq.ns;
    float va[32], vb[32];
    tmem_ld32(taddr, va);
    tmem_wait_ld_dep(va);
    if (t == 0) {
        // visibility is a suffix cut: an all-masked first group means an
        // all-masked row, which gets ref = -inf and contributes nothing
        const int a = rs.a;
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < 30; i += 3)
            mx = max3(mx, fmaxf((skey + i > a) ? -INFINITY : va[i],
                                (skey + i + 1 > a) ? -INFINITY : va[i + 1]),
                      (skey + i + 2 > a) ? -INFINITY : va[i + 2]);
        mx = max3(mx, (skey + 30 > a) ? -INFINITY : va[30], (skey + 31 > a) ? -INFINITY : va[31]);
        rs.ref = mx * s;
        const float bias = (rs.ref == -INFINITY) ? -INFINITY : -rs.ref;
        rs.bias2 = pack2(bias, bias);
    }
#pragma unroll
    for (int cg = 0; cg < kGroups; ++cg) {
        float(&cur)[32] = (cg & 1) ? vb : va;
        float(&nxt)[32] = (cg & 1) ? va : vb;
        if (cg + 1 < kGroups) tmem_ld32(taddr + (cg + 1) * 32, nxt);
        float lo, hi;
        const int kb = skey + cg * 32;
        if (masked) mask_group(cur, kb, rs.a);
        exp_sums(cur, s2, rs.bias2, lo, hi);
        if constexpr (G == 16) {
            const int b = kb / 16;
            st_if(rs.part + (int64_t)b * sq.R, lo, rs.valid && b < sq.nb, rs.policy);
            st_if(rs.part + (int64_t)(b + 1) * sq.R, hi, rs.valid && b + 1 < sq.nb, rs.policy);
            rs.lsum += lo;
            rs.lsum += hi;
        } else {
            rs.acc += lo + hi;
            if ((t * kGroups + cg + 1) % kGroupsPerBlock == 0) {
                const int b = (kb + 32 - G) / G;
                st_if(rs.part + (int64_t)b * sq.R, rs.acc, rs.valid && b < sq.nb, rs.policy);
                rs.lsum += rs.acc;
                rs.acc = 0.f;
            }
        }
        if (cg + 1 < kGroups) {
            tmem_wait_ld_dep(nxt);
            if (cg + 2 == kGroups) {
                // this tile is in registers: hand the buffer back
                tc_fence_before();
                mbar_arrive(smem_u32(&sh.tempty[buf]));
            }
        }
    }
}

// A K step of one row tile, common case: not the unit's first, no key past the
// causal limit (so every block it touches lies inside the sequence).  No
// branch inside, so the compiler can overlap one group's sums with the next
// group's exponentials.  skey is a multiple of 128 and of G when G <= 128; a
// 256-key block closes at the end of every second step of the unit.
// It also tests, without waiting, whether the next slot's TMEM buffer is ready
// (barrier next_bar, phase parity next_par) before its last group's arithmetic,
// so the barrier's latency overlaps that work; the caller skips its own wait
// when next_ready comes back true.
template <int G>
__device__ __forceinline__ void softmax_tile_fast(RowState &rs, uint32_t taddr, int skey, int t,
                                                  int R, uint64_t s2, Shared &sh, int buf,
                                                  uint32_t next_bar, uint32_t next_par,
                                                  bool &next_ready) {
    constexpr int kGroups = kStepKeys / 32;
    constexpr int kGroupsPerBlock = G >= 32 ? G / 32 : 1;
    float *const pb = rs.part + (int64_t)(skey / G) * R;  // the step's first block
    float va[32], vb[32];
    tmem_ld32(taddr, va);
    tmem_wait_ld_dep(va);
#pragma unroll
    for (int cg = 0; cg < kGroups; ++cg) {
        float(&cur)[32] = (cg & 1) ? vb : va;
        float(&nxt)[32] = (cg & 1) ? va : vb;
        if (cg + 1 < kGroups) tmem_ld32(taddr + (cg + 1) * 32, nxt);
        if (cg + 1 == kGroups) next_ready = mbar_test_wait(next_bar, next_par);
        float lo, hi;
        exp_sums(cur, s2, rs.bias2, lo, hi);
        if constexpr (G == 16) {
            st_if(pb + (int64_t)(2 * cg) * R, lo, rs.valid, rs.policy);
            st_if(pb + (int64_t)(2 * cg + 1) * R, hi, rs.valid, rs.policy);
            rs.lsum += lo;
            rs.lsum += hi;
        } else {
            rs.acc += lo + hi;
            const bool closes = G <= 128 ? ((cg + 1) % kGroupsPerBlock == 0)
                                         : (cg + 1 == kGroups && (t & 1));
            if (closes) {
                // the closing block's index relative to the step's first block
                const int off = G <= 128 ? ((cg + 1) * 32 / G - 1) : 0;
                st_if(pb + (int64_t)off * R, rs.acc, rs.valid, rs.policy);
                rs.lsum += rs.acc;
                rs.acc = 0.f;
            }
        }
        if (cg + 1 < kGroups) {
            tmem_wait_ld_dep(nxt);
            if (cg + 2 == kGroups) {
                tc_fence_before();
                mbar_arrive(smem_u32(&sh.tempty[buf]));
            }
        }
    }
}

template <int D, int G>
__device__ void role_softmax(const ScoreParams &p, Shared &sh, uint32_t tmem, int units) {
    using C = Cfg<D>;
    constexpr int kGroups = kStepKeys / 32;
    constexpr int kGroupsPerBlock = G >= 32 ? G / 32 : 1;
    volatile int *abort = &sh.abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = (warp - kWarpEpi) >> 2;  // tile of each pair
    const int quarter = warp & 3;          // TMEM lanes 32*quarter .. +31
    const int row = quarter * 32 + lane;
    // this thread's row of a tile: query tl of the box, head h of the group
    const int tl = row / p.g, h = row - tl * p.g;
    const bool row_used = row < p.g * p.tpt;
    const float s = p.scale_log2;
    const uint64_t s2 = pack2(s, s);
    const uint64_t part_policy = l2_policy_evict_last();
    uint32_t gstep = 0, tpar = 0u;  // bit b: parity of the uses of TMEM buffer b so far
    bool next_ready = false;        // the next slot's buffer was seen ready in advance
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        Unit un;
        decode_unit<D>(p, u, un);
        const SeqInfo &sq = un.sq;
        const int grows = p.g * sq.ns;
        RowState rs[C::kPairs];
#pragma unroll
        for (int pr = 0; pr < C::kPairs; ++pr) {
            const int tile = un.grp * C::kTiles + 2 * pr + e;
            const int tq = tile_box_query(p, sq.ns, tile) + tl;  // query of this row
            rs[pr].valid = row_used && tq >= tile * p.tpt && tq < sq.ns;
            rs[pr].a = sq.L - sq.ns + (rs[pr].valid ? tq : 0);
            rs[pr].r = (int64_t)un.j * grows + (int64_t)tq * p.g + h;
            rs[pr].part = p.part + sq.part_off + rs[pr].r;
            // checked builds: the row's partials and chunk statistics lie in
            // their buffers (otherwise it stores nothing)
            if (rs[pr].valid &&
                !(in_range(sq.part_off + rs[pr].r, (int64_t)(sq.nb - 1) * sq.R + 1, p.part_cap,
                           p.err) &&
                  in_range(sq.stat_off + (int64_t)(kSlotsPerChunk * un.c) * sq.R + rs[pr].r, 1,
                           p.stat_cap, p.err)))
                rs[pr].valid = false;
            rs[pr].policy = part_policy;
            rs[pr].ref = -INFINITY;
            rs[pr].lsum = 0.f;
            rs[pr].acc = 0.f;
            rs[pr].bias2 = 0;
        }
        for (int t = 0; t < un.nsteps; ++t, ++gstep) {
#pragma unroll
            for (int pr = 0; pr < C::kPairs; ++pr) {
                if (pr >= un.npairs) break;
                const int buf = C::kPairs == 2 ? pr : (int)(gstep & 1u);
                const bool ok = next_ready || mbar_wait(smem_u32(&sh.tfull[buf]),
                                                        (tpar >> buf) & 1u, abort, p.wait_limit);
                next_ready = false;
                __syncwarp();  // tcgen05.ld is warp-collective: reconverge after polling
                if (!__all_sync(0xffffffffu, ok)) return;
                tpar ^= 1u << buf;
                tc_fence_after();
                const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) +
                                       (uint32_t)(buf * kBufCols + e * kStepKeys);
                const int skey = un.k0 + t * kStepKeys;
                if (t == 0 || skey + kStepKeys - 1 > sq.L - sq.ns)
                    softmax_tile<G>(un, rs[pr], taddr, t, s2, s, sh, buf);
                else {
                    // the next slot: the unit's next pair, else pair 0 of the next
                    // step or unit (head_dim <= 128); the next step's buffer (256)
                    const int nbuf = C::kPairs == 2 ? (pr + 1 < un.npairs ? pr + 1 : 0)
                                                    : (int)((gstep + 1) & 1u);
                    softmax_tile_fast<G>(rs[pr], taddr, skey, t, sq.R, s2, sh, buf,
                                         smem_u32(&sh.tfull[nbuf]), (tpar >> nbuf) & 1u,
                                         next_ready);
                }
            }
        }
#pragma unroll
        for (int pr = 0; pr < C::kPairs; ++pr) {
            if (pr >= un.npairs) break;
            RowState &st = rs[pr];
            if constexpr (G > 32) {
                // a block cut short by the end of the sequence
                if ((un.nsteps * kGroups) % kGroupsPerBlock != 0) {
                    const int b = (un.k0 + (un.nsteps * kGroups - 1) * 32) / G;
                    if (st.valid && b < sq.nb) st.part[(int64_t)b * sq.R] = st.acc;
                    st.lsum += st.acc;
                    st.acc = 0.f;
                }
            }
            if (st.valid) {
                const int64_t o = sq.stat_off + (int64_t)(kSlotsPerChunk * un.c) * sq.R + st.r;
                p.mref[o] = st.ref;
                p.lsum[o] = st.lsum;
            }
            // fp32 overflow of the sums (logits far above the reference): queue
            // this row tile of the unit for the exact fallback
            const bool bad = st.valid && !(st.lsum <= 3.0e38f);
            if (__any_sync(0xffffffffu, bad) && lane == 0) {
                pdl_wait();  // the plan zeroes the queue counter
                const int idx = atomicAdd(&const_cast<Counters *>(p.counters)->flagged, 1);
                if (idx < p.flag_cap) p.flag_list[idx] = 4 * u + 2 * pr + e;
            }
        }
    }
}

__device__ __forceinline__ int ld_acquire(const int32_t *ptr) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}

__device__ __forceinline__ float dot4(const float4 x, const float4 y, float a) {
    a = fmaf(x.x, y.x, a);
    a = fmaf(x.y, y.y, a);
    a = fmaf(x.z, y.z, a);
    return fmaf(x.w, y.w, a);
}

// Grid barrier of the epilogue: every CTA of the grid arrives (its earlier
// global writes made visible first), then waits for all of them, at most
// wait_limit cycles (then the timeout bit is set and false returned).  The
// grid is at most one CTA per SM, so all of its CTAs are resident together
// unless other work holds SMs for longer than the bound.  Thread 0 also reads
// the overflow queue counter after the first barrier (every tile that will
// ever be queued is queued by then).
__device__ __forceinline__ int grid_barrier(const ScoreParams &p, int32_t *ctr, Shared &sh,
                                            bool read_flags) {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        atomicAdd(ctr, 1);
        const int n = (int)gridDim.x;
        bool ok = ld_acquire(ctr) >= n;
        if (!ok) {
            const long long t0 = clock64();
            while (!(ok = ld_acquire(ctr) >= n))
                if (clock64() - t0 > p.wait_limit) break;
        }
        int st = ok ? 0 : 1;
        if (!ok) atomicOr(p.err, UP_DEVERR_TIMEOUT);
        if (ok && read_flags &&
            *reinterpret_cast<const volatile int32_t *>(&p.counters->flagged) > 0)
            st = 2;
        sh.epi_state = st;
    }
    __syncthreads();
    return sh.epi_state;
}

__device__ __forceinline__ int find_seq_by_row(const SeqInfo *seqs, int B, int64_t r) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (seqs[mid].row_off <= r) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ int find_seq_by_block(const SeqInfo *seqs, int B, int gb) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (seqs[mid].blk_off <= gb) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Epilogue, all threads of every CTA, after the CTA's last unit:
//   barrier 1 -- every unit of the grid is done: all partials and statistics
//                are in memory; if tiles were queued for the exact fallback,
//                the CTAs recompute them (fallback_tiles) and meet at one more
//                barrier;
//   rows      -- a contiguous share of all softmax rows per CTA, kRowLanes
//                threads per row: over the row's key chunks c, the maximum M
//                and normaliser l,
//                  M = max_c mref[c][r],  l = sum_c lsum[c][r] * 2^(mref[c][r] - M),
//                then, in place of mref[c][r], the weight of chunk c's
//                partials, w = 2^(mref[c][r] - M) / (l * n_s * Hq_norm);
//   barrier 2 -- every weight is in memory;
//   blocks    -- a contiguous share of all blocks per CTA, in batches of up to
//                kEpiBlocks blocks of one chunk: score_b = sum_r part[b][r] *
//                w[c(b)][r], thread t taking the float4 groups t, t + 384, ...
//                of the rows in order, then a fixed butterfly and the warps in
//                order -- independent of the grid and the batching, so the
//                scores are bitwise reproducible.
// Loads of other CTAs' results bypass L1.
constexpr int kEpiChunks = 4;   // chunk statistics a thread has in flight (per kRowLanes chunks)
constexpr int kEpiBlocks = 6;   // blocks of one batch (all of their partials in flight)
constexpr int kEpiVec = 3;      // float4 groups per thread and block in flight (rows <= 4608)

// Online merge of a row's (maximum, normaliser) with one chunk's (reference, sum).
__device__ __forceinline__ void merge_chunk(float &M, float &l, float m, float s) {
    if (m == -INFINITY) return;
    if (M == -INFINITY) {
        M = m;
        l = s;
        return;
    }
    const float mn = fmaxf(M, m);
    l = l * exp2f(M - mn) + s * exp2f(m - mn);
    M = mn;
}

// Rows: kRowLanes consecutive threads take one row, each the chunks c = sub,
// sub + kRowLanes, ... (at most kEpiChunks per thread loaded at once); their
// (maximum, normaliser) pairs are merged by a fixed butterfly, so every lane
// ends with the row's M and l (bitwise the same whichever CTA does the row).
constexpr int kRowLanes = 8;

template <int NT>
__device__ void epilogue_rows(const ScoreParams &p) {
    const int64_t total = p.counters->rows;
    const int64_t per = (total + gridDim.x - 1) / gridDim.x;
    const int64_t r0 = (int64_t)blockIdx.x * per, r1 = min(r0 + per, total);
    const int sub = threadIdx.x % kRowLanes;
    constexpr int kRowsPerPass = NT / kRowLanes;
    for (int64_t g0 = r0; g0 < r1; g0 += kRowsPerPass) {
        const int64_t gr = g0 + threadIdx.x / kRowLanes;
        const bool row_ok = gr < r1;
        const SeqInfo &sq = p.num_seqs == 1
                                ? p.seq0
                                : p.seqs[find_seq_by_row(p.seqs, p.num_seqs, row_ok ? gr : r0)];
        const int64_t r = (row_ok ? gr : r0) - sq.row_off;
        float *mref = p.mref + sq.stat_off + r;
        const float *lsum = p.lsum + sq.stat_off + r;
        // checked builds: the row's chunk statistics lie in their buffers
        const bool st_ok = !row_ok || in_range(sq.stat_off + r, (int64_t)(sq.nchunks - 1) * sq.R + 1,
                                               p.stat_cap, p.err);
        const int nch = row_ok && st_ok ? sq.nchunks : 0;
        float M = -INFINITY, l = 0.f;
        // this lane's chunks c = sub + kRowLanes * k; the first kEpiChunks of
        // them stay in registers for the weights
        float m0[kEpiChunks];
#pragma unroll
        for (int k = 0; k < kEpiChunks; ++k) {
            const int c = sub + k * kRowLanes;
            m0[k] = c < nch ? __ldcg(mref + (int64_t)c * sq.R) : -INFINITY;
        }
        {
            float s[kEpiChunks];
#pragma unroll
            for (int k = 0; k < kEpiChunks; ++k) {
                const int c = sub + k * kRowLanes;
                s[k] = c < nch ? __ldcg(lsum + (int64_t)c * sq.R) : 0.f;
            }
#pragma unroll
            for (int k = 0; k < kEpiChunks; ++k) merge_chunk(M, l, m0[k], s[k]);
        }
        for (int c0 = sub + kRowLanes * kEpiChunks; c0 < nch; c0 += kRowLanes * kEpiChunks) {
            float m[kEpiChunks], s[kEpiChunks];
#pragma unroll
            for (int k = 0; k < kEpiChunks; ++k) {
                const int c = c0 + k * kRowLanes;
                m[k] = c < nch ? __ldcg(mref + (int64_t)c * sq.R) : -INFINITY;
                s[k] = c < nch ? __ldcg(lsum + (int64_t)c * sq.R) : 0.f;
            }
#pragma unroll
            for (int k = 0; k < kEpiChunks; ++k) merge_chunk(M, l, m[k], s[k]);
        }
#pragma unroll
        for (int o = 1; o < kRowLanes; o <<= 1) {
            const float Mo = __shfl_xor_sync(0xffffffffu, M, o);
            const float lo = __shfl_xor_sync(0xffffffffu, l, o);
            // the lower lane's pair first, so both lanes compute the same bits
            if ((sub & o) == 0) merge_chunk(M, l, Mo, lo);
            else {
                float M2 = Mo, l2 = lo;
                merge_chunk(M2, l2, M, l);
                M = M2;
                l = l2;
            }
        }
        const float inv = (M == -INFINITY || !(l > 0.f))
                              ? 0.f
                              : 1.0f / (l * (float)sq.ns * (float)p.Hq_norm);
        auto weight = [&](float m) { return (m == -INFINITY || inv == 0.f) ? 0.f : exp2f(m - M) * inv; };
#pragma unroll
        for (int k = 0; k < kEpiChunks; ++k) {
            const int c = sub + k * kRowLanes;
            if (c < nch) mref[(int64_t)c * sq.R] = weight(m0[k]);
        }
        for (int c = sub + kRowLanes * kEpiChunks; c < nch; c += kRowLanes) {
            float *q = mref + (int64_t)c * sq.R;
            *q = weight(__ldcg(q));
        }
    }
}

template <int NT>
__device__ void epilogue_blocks(const ScoreParams &p, float (*red)[NT / 32]) {
    constexpr int kWarps = NT / 32;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int nbt = p.counters->blocks;
    const int per = (nbt + (int)gridDim.x - 1) / (int)gridDim.x;
    const int lo = (int)blockIdx.x * per, hi = min(lo + per, nbt);
    if (lo >= hi) return;
    const int bpc = p.C / p.G;  // blocks per key chunk
    int s = p.num_seqs == 1 ? 0 : find_seq_by_block(p.seqs, p.num_seqs, lo);
    for (int gb = lo; gb < hi;) {
        if (p.num_seqs != 1)
            while (gb >= p.seqs[s].blk_off + p.seqs[s].nb) ++s;  // skips empty sequences
        const SeqInfo &sq = p.num_seqs == 1 ? p.seq0 : p.seqs[s];
        const int b = gb - sq.blk_off;
        const int nbat = min(min(kEpiBlocks, hi - gb), min(sq.nb - b, (b / bpc + 1) * bpc - b));
        const float *wr = p.mref + sq.stat_off + (int64_t)block_slot(b, p.G, p.C) * sq.R;
        const float *pt = p.part + sq.part_off + (int64_t)b * sq.R;
        // checked builds: the batch's partials, weights and scores lie in their
        // buffers (the test is the same in every thread of the CTA)
        if (!(in_range(sq.part_off + (int64_t)b * sq.R, (int64_t)nbat * sq.R, p.part_cap, p.err) &&
              in_range(sq.stat_off + (int64_t)block_slot(b, p.G, p.C) * sq.R, sq.R, p.stat_cap,
                       p.err) &&
              in_range(gb, nbat, p.scores_cap, p.err))) {
            gb += nbat;
            continue;
        }
        float acc[kEpiBlocks];
#pragma unroll
        for (int k = 0; k < kEpiBlocks; ++k) acc[k] = 0.f;
        if ((sq.R % 4 == 0) && ((sq.stat_off | sq.part_off) % 4 == 0)) {
            const float4 *w4 = reinterpret_cast<const float4 *>(wr);
            const float4 *p4 = reinterpret_cast<const float4 *>(pt);
            const int R4 = sq.R / 4;
            const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int i0 = threadIdx.x; i0 < R4; i0 += kEpiVec * NT) {
                float4 w[kEpiVec], x[kEpiBlocks][kEpiVec];
#pragma unroll
                for (int u = 0; u < kEpiVec; ++u) {
                    const int i = i0 + u * NT;
                    w[u] = i < R4 ? __ldcg(w4 + i) : zero;
                }
#pragma unroll
                for (int k = 0; k < kEpiBlocks; ++k)
#pragma unroll
                    for (int u = 0; u < kEpiVec; ++u) {
                        const int i = i0 + u * NT;
                        x[k][u] = (k < nbat && i < R4) ? __ldcg(p4 + (int64_t)k * R4 + i) : zero;
                    }
#pragma unroll
                for (int k = 0; k < kEpiBlocks; ++k)
#pragma unroll
                    for (int u = 0; u < kEpiVec; ++u) acc[k] = dot4(x[k][u], w[u], acc[k]);
            }
        } else {
            for (int r = threadIdx.x; r < sq.R; r += NT) {
                const float w = __ldcg(wr + r);
#pragma unroll
                for (int k = 0; k < kEpiBlocks; ++k)
                    if (k < nbat) acc[k] = fmaf(__ldcg(pt + (int64_t)k * sq.R + r), w, acc[k]);
            }
        }
#pragma unroll
        for (int k = 0; k < kEpiBlocks; ++k) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], o);
        }
        if (lane == 0) {
#pragma unroll
            for (int k = 0; k < kEpiBlocks; ++k) red[k][wid] = acc[k];
        }
        __syncthreads();
        if ((int)threadIdx.x < nbat) {
            float t = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) t += red[threadIdx.x][w];
            p.scores[gb + threadIdx.x] = t;
        }
        __syncthreads();
        gb += nbat;
    }
}

// The exact fallback for the rare row tiles whose fp32 sums overflowed in the
// main loop: a logit more than ~115 binary orders of magnitude above the
// unit's reference (taken from its first 32 keys).  Each queued tile (4 *
// unit + tile) is recomputed by one CTA on the CUDA cores with two passes over
// the unit's keys: the first finds each row's exact maximum m (log2 units),
// the second sums 2^(z*log2e/sqrt(d) - m) over every block; the tile's
// partials and chunk statistics are rewritten.  Row r of the tile is thread r
// (128 of the CTA's threads compute; all of them stage Q and K in shared
// memory).  The queue is empty for ordinary attention logits.
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
__device__ void fallback_tiles(const ScoreParams &p, unsigned char *smem) {
    const int nflag =
        min(*reinterpret_cast<const volatile int32_t *>(&p.counters->flagged), p.flag_cap);
    __nv_bfloat16 *qT = reinterpret_cast<__nv_bfloat16 *>(smem);         // [D][128]
    float *ks = reinterpret_cast<float *>(smem + D * kRowsPerTile * 2);  // [32][D]
    const int tid = threadIdx.x;
    const bool row_thread = tid < kRowsPerTile;
    for (int fi = blockIdx.x; fi < nflag; fi += gridDim.x) {
        const int entry = __ldcg(p.flag_list + fi);
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
        const bool valid = row_thread && tid < p.g * p.tpt && t < sq.ns &&
                           in_range(sq.part_off + (int64_t)j * grows + (int64_t)t * p.g + h,
                                    (int64_t)(sq.nb - 1) * sq.R + 1, p.part_cap, p.err) &&
                           in_range(sq.stat_off + (int64_t)(kSlotsPerChunk * c) * sq.R +
                                        (int64_t)j * grows + (int64_t)t * p.g + h,
                                    1, p.stat_cap, p.err);
        const int a = sq.L - sq.ns + (valid ? t : 0);
        const int64_t r = (int64_t)j * grows + (int64_t)t * p.g + h;
        __syncthreads();
        for (int idx = tid; idx < kRowsPerTile * D; idx += Cfg<D>::kThreads) {
            const int row = idx / D, cc = idx % D;
            const int rtl = row / p.g, rh = row - rtl * p.g, rt = mt * p.tpt + rtl;
            __nv_bfloat16 v = __float2bfloat16(0.f);
            if (row < p.g * p.tpt && rt < sq.ns)
                v = p.q[((int64_t)(sq.q_off + rt) * p.Hq + j * p.g + rh) * D + cc];
            qT[cc * kRowsPerTile + row] = v;
        }
        const int k0 = c * p.C;
        const int k1 = min(k0 + p.C, sq.L);
        float m = -INFINITY, lsum = 0.f;
        float acc[kKeyTile];
        for (int pass = 0; pass < 2; ++pass) {
            float bsum = 0.f;
            for (int kt = k0; kt < k1; kt += kKeyTile) {
                __syncthreads();
                for (int idx = tid; idx < kKeyTile * D; idx += Cfg<D>::kThreads) {
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
                if (!row_thread) continue;
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
__device__ void score_epilogue(const ScoreParams &p, Shared &sh, float *smem_f) {
    pdl_wait();  // the plan's table and counters
    Counters *cnt = const_cast<Counters *>(p.counters);
    const int st = grid_barrier(p, &cnt->bar[0], sh, true);
    if (st == 1) return;  // a wait expired
    if (st == 2) {
        // tiles overflowed: recompute them exactly before the rows read them
        fallback_tiles<D>(p, reinterpret_cast<unsigned char *>(smem_f));
        if (grid_barrier(p, &cnt->bar[2], sh, false) != 0) return;
    }
    epilogue_rows<Cfg<D>::kThreads>(p);
    if (grid_barrier(p, &cnt->bar[1], sh, false) != 0) return;
    epilogue_blocks<Cfg<D>::kThreads>(
        p, reinterpret_cast<float(*)[Cfg<D>::kThreads / 32]>(smem_f));
}

template <int D, int G>
__global__ void __launch_bounds__(Cfg<D>::kThreads, 1)
score_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                const ScoreParams p) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ Shared sh;
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *qbuf = smem;                          // Q buffers (1024-aligned panels)
    uint8_t *kbuf = smem + C::kQBufs * C::kQBytes; // kStages x K panel
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        // One sequence: the work is known from the host's sizes once cu_seqlens
        // is confirmed to be {0, total}, and nothing below needs the plan (the
        // kernels before it are complete).  Otherwise wait for the plan's table.
        if (p.num_seqs == 1) {
            const bool ok = p.cu_seqlens[0] == 0 && p.cu_seqlens[1] == p.seq0.L;
            sh.units = ok ? p.units0 : 0;
        } else {
            pdl_wait();
            sh.units = p.counters->units;
        }
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(smem_u32(&sh.kfull[i]), 1);
            mbar_init(smem_u32(&sh.kempty[i]), C::kStageUsers);
        }
        for (int q = 0; q < C::kQSlots; ++q) {
            mbar_init(smem_u32(&sh.qfull[q]), 1);
            mbar_init(smem_u32(&sh.qempty[q]), C::kQUsers);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&sh.tfull[b]), 2);  // one commit per issuer
            mbar_init(smem_u32(&sh.tempty[b]), 2 * kEpiThreads);
            mbar_init(smem_u32(&sh.fin[b]), 1);
        }
        sh.abort = 0;
        sh.epi_state = 0;
        fence_mbar_init();
    }
    if (warp == kWarpMma0) {
        tmem_alloc(smem_u32(&sh.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    if (warp == kWarpTmaK && lane == 0) {
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&qmap);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    const int units = sh.units;
    if (p.num_seqs != 1) pdl_wait();  // every thread past the plan before reading its table

    if (warp == kWarpTmaK) {
        if (lane == 0) role_tma_k<D>(&kmap, p, sh, kbuf, units);
    } else if (warp == kWarpTmaQ) {
        if (lane == 0) role_tma_q<D>(&qmap, p, sh, qbuf, units);
    } else if (warp == kWarpMma0 || warp == kWarpMma1) {
        role_mma<D>(p, sh, qbuf, kbuf, tmem, units, warp == kWarpMma0 ? 0 : 1);
    } else {
        role_softmax<D, G>(p, sh, tmem, units);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (!sh.abort) {
        // the epilogue's generic stores reuse shared memory the TMA wrote
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        score_epilogue<D>(p, sh, reinterpret_cast<float *>(smem));
    }
    if (threadIdx.x == 0 && sh.abort) atomicOr(p.err, UP_DEVERR_TIMEOUT);
    pdl_wait();  // this grid completes after the plan: later kernels read its table
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// K viewed as a 2-D row-major matrix [total_tokens, Hk*d] (paged keys:
// [num_pages*Hk*page_size, d]); one box = 128 rows (keys) x 64 columns (head
// dims) with the 128-byte swizzle.  Rows past the end read as zeros.
bool encode_k_map(CUtensorMap *tm, const ScoreParams &p, int64_t total_tokens) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    // paged keys: [num_pages * Hk * page_size rows, d], the same 128 x 64 box
    const bool paged = p.block_table != nullptr;
    const cuuint64_t dims[2] = {
        (cuuint64_t)(paged ? p.d : p.Hk * p.d),
        (cuuint64_t)(paged ? p.num_pages * p.Hk * p.page_size : total_tokens)};
    const cuuint64_t strides[1] = {(cuuint64_t)(paged ? p.d : p.Hk * p.d) * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kStepKeys};
    const cuuint32_t estr[2] = {1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16 *>(p.k), dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// q_last viewed as a 3-D array [queries][Hq][d] (d innermost); one box = 64 head
// dims x g query heads x tpt queries, with the 128-byte swizzle.  The query
// extent is an upper bound on the rows of q_last (the exact count is only known
// on the device); the kernel never addresses a query past its own sequence, and
// coordinates below 0 read as zeros.
bool encode_q_map(CUtensorMap *tm, const ScoreParams &p, int64_t max_qrows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)p.d, (cuuint64_t)p.Hq,
                                (cuuint64_t)(max_qrows > 0 ? max_qrows : 1)};
    const cuuint64_t strides[2] = {(cuuint64_t)p.d * 2, (cuuint64_t)p.Hq * p.d * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)p.g, (cuuint32_t)p.tpt};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<__nv_bfloat16 *>(p.q), dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int G>
cudaError_t launch_dg(const ScoreParams &p, const ScoreLayout &lay, int num_sms, cudaStream_t st) {
    CUtensorMap km, qm;
    if (!encode_k_map(&km, p, lay.total_tokens)) return cudaErrorInvalidValue;
    if (!encode_q_map(&qm, p, lay.max_qrows)) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(score_tc_kernel<D, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::kSmem);
    if (e != cudaSuccess) return e;
    const int64_t grid = lay.max_units < num_sms ? lay.max_units : num_sms;
    if (grid < 1) return cudaSuccess;
    return launch_pdl(score_tc_kernel<D, G>, dim3((unsigned)grid), dim3(Cfg<D>::kThreads),
                      Cfg<D>::kSmem, st,
                      km, qm, p);
}

template <int D>
cudaError_t launch_d(const ScoreParams &p, const ScoreLayout &lay, int num_sms, cudaStream_t st) {
    switch (p.G) {
        case 16: return launch_dg<D, 16>(p, lay, num_sms, st);
        case 32: return launch_dg<D, 32>(p, lay, num_sms, st);
        case 64: return launch_dg<D, 64>(p, lay, num_sms, st);
        case 128: return launch_dg<D, 128>(p, lay, num_sms, st);
        case 256: return launch_dg<D, 256>(p, lay, num_sms, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_score_main(const ScoreParams &p, const ScoreLayout &lay, int num_sms,
                              cudaStream_t st) {
    switch (p.d) {
        case 64: return launch_d<64>(p, lay, num_sms, st);
        case 128: return launch_d<128>(p, lay, num_sms, st);
        case 256: return launch_d<256>(p, lay, num_sms, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace up
