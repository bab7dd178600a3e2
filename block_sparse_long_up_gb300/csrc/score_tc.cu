// score_tc.cu -- block scoring on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// UniPrefill overview, block-wise importance estimation paragraph: the last n
// queries of a sequence are dotted with all of its keys, the softmax mass of
// each query is summed over fixed blocks of G keys and averaged over queries
// and heads.  Its fused-kernel paragraph names the pieces fused here: loads from
// HBM, online softmax and block reduction in one pipeline.
//
// Work unit = (sequence s, KV head j, pair of 128-row tiles, key chunk c).  The
// rows are the packed GQA rows r = (query head h of group j, query t), so one K
// step serves every query head that shares it (the PackGQA idea of the
// FlashPrefill V2 review, re-derived for tcgen05), and one K panel in shared
// memory feeds both row tiles, halving the K bytes each SM must stream per MMA.
// A persistent CTA per SM walks its units; roles are warp-specialised:
//   warp 0      TMA producer: 128-key x 64-dim K panels (128-byte swizzle) into
//               a ring of shared-memory stages;
//   warp 1      TMEM owner and MMA issuer: for each 128-key step, S = Q K^T for
//               both row tiles (M=128, N=128 tcgen05.mma chains) into one of two
//               TMEM buffers (2 steps x 2 tiles x 128 fp32 columns = 512);
//   warps 2-3   Q loader: the unit's 256 packed query rows, swizzled into a
//               K-major tile (double-buffered when shared memory allows);
//   warps 4-11  two softmax warpgroups; warpgroup e owns row tile e.  Thread =
//               row (TMEM lane).  It reads 32 columns at a time (the next
//               group's TMEM load in flight while the current one is processed),
//               applies the causal mask on the last steps, computes
//               2^(z*log2e/sqrt(d) - ref) -- most on the MUFU, a fixed share with
//               an FMA-pipe polynomial -- and sums each block of G keys; the
//               block sums go straight to HBM as partials.
// The reference `ref` of a row is the largest visible logit among the first 32
// keys of the unit; the row's statistics for the chunk (ref and the sum of all
// its block partials) go to workspace.  Later keys may exceed ref; fp32 absorbs
// that up to ~115 binary orders of magnitude, and a tile whose sums overflow
// anyway is queued for the exact CUDA-core fallback.
#include <cudaTypedefs.h>

#include "../../include/up.h"
#include "common.cuh"
#include "sm100.cuh"

namespace up {

namespace {

using namespace sm100;

constexpr int kThreads = 384;
constexpr int kWarpTma = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpQ = 2;        // warps 2 and 3
constexpr int kQThreads = 64;
constexpr int kWarpEpi = 4;      // warps 4..11: two warpgroups
constexpr int kEpiThreads = 128; // one warpgroup
constexpr int kPanelBytesK = kStepKeys * 128;      // 128 keys x 64 bf16 = 16 KB
constexpr int kPanelBytesQ = kRowsPerTile * 128;   // 128 rows x 64 bf16 = 16 KB
constexpr uint32_t kTmemCols = 512;
constexpr int kSmemBudget = 227 * 1024 - 2048;     // dynamic bytes we allow ourselves
constexpr long long kWaitLimit = 4000000000LL;     // cycles, ~2 s
constexpr int kMaxStages = 16;

template <int D>
struct Cfg {
    static constexpr int kPanels = D / 64;
    static constexpr int kQTileBytes = kPanels * kPanelBytesQ;           // one row tile
    static constexpr int kQBytes = kTilesPerUnit * kQTileBytes;          // one Q buffer
    static constexpr int kQBufs = (2 * kQBytes + 6 * kPanelBytesK <= kSmemBudget) ? 2 : 1;
    static constexpr int kStagesFit = (kSmemBudget - 1024 - kQBufs * kQBytes) / kPanelBytesK;
    static constexpr int kStages = kStagesFit < kMaxStages ? kStagesFit : kMaxStages;
    static constexpr int kSmem = kQBufs * kQBytes + kStages * kPanelBytesK + 1024;
    static_assert(kStages >= kPanels, "at least one K step in flight");
};

struct Shared {
    uint64_t kfull[kMaxStages], kempty[kMaxStages];
    uint64_t qfull[2], qempty[2];
    uint64_t tfull[2], tempty[2];
    uint64_t fin;
    uint32_t tmem_base;
    int abort;
};

struct Unit {
    SeqInfo sq;
    int j, mp, c, k0, k1, nsteps;
};

__device__ __forceinline__ void decode_unit(const ScoreParams &p, int u, Unit &un) {
    const int s = find_seq_by_unit(p.seqs, p.num_seqs, u);
    un.sq = p.seqs[s];
    int loc = u - un.sq.unit_off;
    un.mp = loc % un.sq.mtiles;  // row-tile pair
    loc /= un.sq.mtiles;
    un.c = loc % un.sq.nchunks;
    un.j = loc / un.sq.nchunks;
    un.k0 = un.c * p.C;
    un.k1 = min(un.k0 + p.C, un.sq.L);
    un.nsteps = (un.k1 - un.k0 + kStepKeys - 1) / kStepKeys;
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
__device__ void role_tma(const CUtensorMap *tmap, const ScoreParams &p, Shared &sh,
                         uint8_t *kbuf, int units) {
    using C = Cfg<D>;
    volatile int *abort = &sh.abort;
    uint32_t it = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        Unit un;
        decode_unit(p, u, un);
        for (int t = 0; t < un.nsteps; ++t) {
            const int row0 = un.sq.tok_off + un.k0 + t * kStepKeys;
            for (int pn = 0; pn < C::kPanels; ++pn, ++it) {
                const int st = it % C::kStages;
                const uint32_t ph = (it / C::kStages) & 1;
                if (!mbar_wait(smem_u32(&sh.kempty[st]), ph ^ 1, abort, kWaitLimit)) goto aborted;
                mbar_arrive_expect_tx(smem_u32(&sh.kfull[st]), kPanelBytesK);
                tma_load_2d(smem_u32(kbuf + st * kPanelBytesK), tmap, un.j * D + pn * 64, row0,
                            smem_u32(&sh.kfull[st]));
            }
        }
    }
    return;
aborted:
    // let the loads already issued land before the CTA can exit
    for (uint32_t k = 0; k < (uint32_t)C::kStages && k < it; ++k) {
        const uint32_t i = it - 1 - k;
        mbar_drain(smem_u32(&sh.kfull[i % C::kStages]), (i / C::kStages) & 1);
    }
}

template <int D>
__device__ void role_qload(const ScoreParams &p, Shared &sh, uint8_t *qbuf, int units) {
    using C = Cfg<D>;
    constexpr int kCh = D / 8;  // 16-byte chunks per row
    constexpr int kTotal = kTilesPerUnit * kRowsPerTile * kCh;
    constexpr int kBatch = 8;
    volatile int *abort = &sh.abort;
    const int qt = threadIdx.x - kWarpQ * 32;
    uint32_t ui = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++ui) {
        Unit un;
        decode_unit(p, u, un);
        const int qb = ui % C::kQBufs;
        const uint32_t use = ui / C::kQBufs;
        if (!mbar_wait(smem_u32(&sh.qempty[qb]), (use & 1) ^ 1, abort, kWaitLimit)) return;
        uint8_t *dst = qbuf + qb * C::kQBytes;
        const int ns = un.sq.ns;
        const int grows = p.g * ns;
        const int row_base = un.mp * kTilesPerUnit * kRowsPerTile;
        for (int base = qt; base < kTotal; base += kQThreads * kBatch) {
            uint4 v[kBatch];
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                const int idx = base + i * kQThreads;
                v[i] = make_uint4(0, 0, 0, 0);
                if (idx < kTotal) {
                    const int row = idx / kCh, ch = idx % kCh;
                    const int rr = row_base + row;
                    if (rr < grows) {
                        const int hh = rr / ns, tt = rr % ns;
                        const __nv_bfloat16 *src =
                            p.q + ((int64_t)(un.sq.q_off + tt) * p.Hq + un.j * p.g + hh) * D + ch * 8;
                        v[i] = __ldg(reinterpret_cast<const uint4 *>(src));
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                const int idx = base + i * kQThreads;
                if (idx < kTotal) {
                    const int row = idx / kCh, ch = idx % kCh;
                    const int tile = row / kRowsPerTile, tr = row % kRowsPerTile;
                    const int pn = ch >> 3, c16 = ch & 7;
                    uint8_t *d = dst + tile * C::kQTileBytes + pn * kPanelBytesQ + tr * 128 +
                                 ((c16 ^ (tr & 7)) << 4);
                    *reinterpret_cast<uint4 *>(d) = v[i];
                }
            }
        }
        fence_proxy_async_smem();
        mbar_arrive(smem_u32(&sh.qfull[qb]));
    }
}

template <int D>
__device__ void role_mma(const ScoreParams &p, Shared &sh, uint8_t *qbuf, uint8_t *kbuf,
                         uint32_t tmem, int units) {
    using C = Cfg<D>;
    constexpr uint32_t idesc = idesc_bf16_f32(kRowsPerTile, kStepKeys);
    volatile int *abort = &sh.abort;
    uint32_t it = 0, step = 0, ui = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++ui) {
        Unit un;
        decode_unit(p, u, un);
        const int qb = ui % C::kQBufs;
        if (!mbar_wait(smem_u32(&sh.qfull[qb]), (ui / C::kQBufs) & 1, abort, kWaitLimit)) goto out;
        tc_fence_after();
        {
            const uint32_t qaddr = smem_u32(qbuf + qb * C::kQBytes);
            for (int t = 0; t < un.nsteps; ++t, ++step) {
                const int b = step & 1;
                if (!mbar_wait(smem_u32(&sh.tempty[b]), ((step >> 1) & 1) ^ 1, abort, kWaitLimit))
                    goto out;
                tc_fence_after();
                for (int pn = 0; pn < C::kPanels; ++pn, ++it) {
                    const int st = it % C::kStages;
                    if (!mbar_wait(smem_u32(&sh.kfull[st]), (it / C::kStages) & 1, abort, kWaitLimit))
                        goto out;
                    tc_fence_after();
                    const uint64_t bd = smem_desc_sw128(smem_u32(kbuf + st * kPanelBytesK));
#pragma unroll
                    for (int e = 0; e < kTilesPerUnit; ++e) {
                        const uint32_t d_tmem =
                            tmem + (uint32_t)(b * kTilesPerUnit * kStepKeys + e * kStepKeys);
                        const uint64_t ad =
                            smem_desc_sw128(qaddr + e * C::kQTileBytes + pn * kPanelBytesQ);
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)  // 4 x K=16 per 64-wide panel (32 B each)
                            mma_bf16(d_tmem, ad + 2 * ks, bd + 2 * ks, idesc, (pn | ks) != 0);
                    }
                    mma_commit(smem_u32(&sh.kempty[st]));
                }
                mma_commit(smem_u32(&sh.tfull[b]));
            }
        }
        mma_commit(smem_u32(&sh.qempty[qb]));
    }
out:
    // every MMA issued by this thread has completed once fin fires
    mma_commit(smem_u32(&sh.fin));
    mbar_drain(smem_u32(&sh.fin), 0);
}

// One 32-column group: scale, mask, exponentiate, and sum the two 16-column
// halves.  Lane pairs (i, i+16) share one packed register so that the fixed
// summation tree ends with (sum of columns 0..15, sum of 16..31).  Pairs 0..2
// (6 of 32 values) are exponentiated on the FMA pipe, the rest on the MUFU.
constexpr int kPolyPairs = 3;

__device__ __forceinline__ void group_exp_sums(float (&v)[32], bool masked, int key, int a,
                                               uint64_t s2, uint64_t bias2, float &lo, float &hi) {
    if (masked) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = (key + i > a) ? -INFINITY : v[i];
    }
    uint64_t x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint64_t z = fma2(pack2(v[i], v[i + 16]), s2, bias2);
        float z0, z1;
        unpack2(z, z0, z1);
        x[i] = (i < kPolyPairs) ? ex2_poly2(z0, z1) : pack2(ex2_approx(z0), ex2_approx(z1));
    }
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1) {
#pragma unroll
        for (int i = 0; i < w; ++i) x[i] = add2(x[2 * i], x[2 * i + 1]);
    }
    unpack2(x[0], lo, hi);
}

template <int D, int G>
__device__ void role_softmax(const ScoreParams &p, Shared &sh, uint32_t tmem, int units) {
    constexpr int kGroups = kStepKeys / 32;
    constexpr int kGroupsPerBlock = G >= 32 ? G / 32 : 1;
    volatile int *abort = &sh.abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = (warp - kWarpEpi) >> 2;  // row tile of the pair
    const int quarter = warp & 3;          // TMEM lanes 32*quarter .. +31
    const int row = quarter * 32 + lane;
    const float s = p.scale_log2;
    const uint64_t s2 = pack2(s, s);
    uint32_t step = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        Unit un;
        decode_unit(p, u, un);
        const SeqInfo &sq = un.sq;
        const int grows = p.g * sq.ns;
        const int rl = (un.mp * kTilesPerUnit + e) * kRowsPerTile + row;
        const bool valid = rl < grows;
        const int a = sq.L - sq.ns + (valid ? rl % sq.ns : 0);  // causal limit of this row
        const int64_t r = (int64_t)un.j * grows + rl;           // h * n_s + t
        float *part = p.part + sq.part_off + r;
        float lsum = 0.f, ref = -INFINITY, acc = 0.f;
        uint64_t bias2 = 0;
        for (int t = 0; t < un.nsteps; ++t, ++step) {
            const int buf = step & 1;
            const bool ok = mbar_wait(smem_u32(&sh.tfull[buf]), (step >> 1) & 1, abort, kWaitLimit);
            __syncwarp();  // tcgen05.ld is warp-collective: reconverge after polling
            if (!__all_sync(0xffffffffu, ok)) return;
            tc_fence_after();
            const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) +
                                   (uint32_t)(buf * kTilesPerUnit * kStepKeys + e * kStepKeys);
            const int skey = un.k0 + t * kStepKeys;  // first key of the step
            const bool masked = skey + kStepKeys - 1 > sq.L - sq.ns;
            float va[32], vb[32];
            tmem_ld32(taddr, va);
            tmem_wait_ld_dep(va);
            if (t == 0) {
                // visibility is a suffix cut: an all-masked first group means an
                // all-masked row, which gets ref = -inf and contributes nothing
                float mx = -INFINITY;
#pragma unroll
                for (int i = 0; i < 30; i += 3)
                    mx = max3(mx, fmaxf((skey + i > a) ? -INFINITY : va[i],
                                        (skey + i + 1 > a) ? -INFINITY : va[i + 1]),
                              (skey + i + 2 > a) ? -INFINITY : va[i + 2]);
                mx = max3(mx, (skey + 30 > a) ? -INFINITY : va[30],
                          (skey + 31 > a) ? -INFINITY : va[31]);
                ref = mx * s;
                const float bias = (ref == -INFINITY) ? -INFINITY : -ref;
                bias2 = pack2(bias, bias);
            }
#pragma unroll
            for (int cg = 0; cg < kGroups; ++cg) {
                float(&cur)[32] = (cg & 1) ? vb : va;
                float(&nxt)[32] = (cg & 1) ? va : vb;
                if (cg + 1 < kGroups) tmem_ld32(taddr + (cg + 1) * 32, nxt);
                float lo, hi;
                const int kb = skey + cg * 32;
                group_exp_sums(cur, masked, kb, a, s2, bias2, lo, hi);
                if constexpr (G == 16) {
                    const int b = kb / 16;
                    if (valid && b < sq.nb) part[(int64_t)b * sq.R] = lo;
                    if (valid && b + 1 < sq.nb) part[(int64_t)(b + 1) * sq.R] = hi;
                    lsum += lo;
                    lsum += hi;
                } else {
                    acc += lo + hi;
                    if ((t * kGroups + cg + 1) % kGroupsPerBlock == 0) {
                        const int b = (kb + 32 - G) / G;
                        if (valid && b < sq.nb) part[(int64_t)b * sq.R] = acc;
                        lsum += acc;
                        acc = 0.f;
                    }
                }
                if (cg + 1 < kGroups) {
                    tmem_wait_ld_dep(nxt);
                    if (cg + 2 == kGroups) {
                        // this tile of the step is in registers: hand the buffer back
                        tc_fence_before();
                        mbar_arrive(smem_u32(&sh.tempty[buf]));
                    }
                }
            }
        }
        if constexpr (G > 32) {
            // a block cut short by the end of the sequence
            if ((un.nsteps * kGroups) % kGroupsPerBlock != 0) {
                const int b = (un.k0 + (un.nsteps * kGroups - 1) * 32) / G;
                if (valid && b < sq.nb) part[(int64_t)b * sq.R] = acc;
                lsum += acc;
                acc = 0.f;
            }
        }
        if (valid) {
            const int64_t o = sq.stat_off + (int64_t)(kSlotsPerChunk * un.c) * sq.R + r;
            p.mref[o] = ref;
            p.lsum[o] = lsum;
        }
        // fp32 overflow of the sums (logits far above the reference): queue this
        // row tile of the unit for the exact fallback
        const bool bad = valid && !(lsum <= 3.0e38f);
        if (__any_sync(0xffffffffu, bad) && lane == 0) {
            const int idx = atomicAdd(&const_cast<Counters *>(p.counters)->flagged, 1);
            if (idx < p.flag_cap) p.flag_list[idx] = 2 * u + e;
        }
    }
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
score_tc_kernel(const __grid_constant__ CUtensorMap tmap, const ScoreParams p) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ Shared sh;
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *qbuf = smem;                          // Q buffers (1024-aligned panels)
    uint8_t *kbuf = smem + C::kQBufs * C::kQBytes; // kStages x K panel
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int units = p.counters->units;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(smem_u32(&sh.kfull[i]), 1);
            mbar_init(smem_u32(&sh.kempty[i]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&sh.qfull[b]), kQThreads);
            mbar_init(smem_u32(&sh.qempty[b]), 1);
            mbar_init(smem_u32(&sh.tfull[b]), 1);
            mbar_init(smem_u32(&sh.tempty[b]), kTilesPerUnit * kEpiThreads);
        }
        mbar_init(smem_u32(&sh.fin), 1);
        sh.abort = 0;
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_u32(&sh.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    if (warp == kWarpTma && lane == 0) tma_prefetch_desc(&tmap);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;

    if (warp == kWarpTma) {
        if (lane == 0) role_tma<D>(&tmap, p, sh, kbuf, units);
    } else if (warp == kWarpMma) {
        if (lane == 0) role_mma<D>(p, sh, qbuf, kbuf, tmem, units);
    } else if (warp < kWarpEpi) {
        role_qload<D>(p, sh, qbuf, units);
    } else {
        role_softmax<D, G>(p, sh, tmem, units);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (threadIdx.x == 0 && sh.abort) atomicOr(p.err, UP_DEVERR_TIMEOUT);
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

// K viewed as a 2-D row-major matrix [total_tokens, Hk*d]; one box = 128 rows
// (keys) x 64 columns (head dims) with the 128-byte swizzle.  Rows past the end
// read as zeros.
bool encode_k_map(CUtensorMap *tm, const ScoreParams &p, int64_t total_tokens) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)p.Hk * p.d, (cuuint64_t)total_tokens};
    const cuuint64_t strides[1] = {(cuuint64_t)p.Hk * p.d * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kStepKeys};
    const cuuint32_t estr[2] = {1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16 *>(p.k), dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int G>
cudaError_t launch_dg(const ScoreParams &p, const ScoreLayout &lay, int num_sms, cudaStream_t st) {
    CUtensorMap tm;
    if (!encode_k_map(&tm, p, lay.total_tokens)) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(score_tc_kernel<D, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::kSmem);
    if (e != cudaSuccess) return e;
    const int64_t grid = lay.max_units < num_sms ? lay.max_units : num_sms;
    if (grid < 1) return cudaSuccess;
    score_tc_kernel<D, G><<<(unsigned)grid, kThreads, Cfg<D>::kSmem, st>>>(tm, p);
    return cudaGetLastError();
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
