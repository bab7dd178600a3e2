// score_tc.cu -- block scoring on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// UniPrefill overview, block-wise importance estimation paragraph: the last n
// queries of a sequence are dotted with all of its keys, the softmax mass of
// each query is summed over fixed blocks of G keys and averaged over queries
// and heads.  Its fused-kernel paragraph names the pieces fused here: loads from
// HBM, online softmax and block reduction in one pipeline.
//
// Work unit = (sequence s, KV head j, 128-row tile mt, key chunk c).  The 128
// rows are the packed GQA rows r = (query head h of group j, query t), so one
// K tile serves all query heads that share it (the PackGQA idea of the
// FlashPrefill V2 review, re-derived for tcgen05).  A persistent CTA per SM
// walks its units; roles are warp-specialised:
//   warp 0      TMA producer: 256-key x 64-dim K panels (128-byte swizzle) into
//               a ring of shared-memory stages;
//   warp 1      TMEM owner and MMA issuer: S = Q K^T for one 128 x 256 tile
//               per tcgen05.mma chain into one of two TMEM accumulators
//               (2 x 256 fp32 columns);
//   warps 2-3   Q loader: the unit's 128 packed query rows, swizzled into a
//               double-buffered K-major tile;
//   warps 4-11  two softmax warpgroups; warpgroup w takes every other tile
//               (TMEM buffer w).  Thread = row (TMEM lane).  For each tile it
//               reads 32 columns at a time, applies the causal mask on the
//               last tiles, computes 2^(z*log2e/sqrt(d) - ref) and sums the
//               values of each block of G keys; the block sums go straight to
//               HBM as partials.
// The reference `ref` of a warpgroup is the exact maximum of its first tile in
// the unit; the unit's statistics (ref and the sum of all its block partials)
// go to the warpgroup's slot.  Later tiles may exceed ref; fp32 absorbs that up
// to ~115 binary orders of magnitude, and a unit whose sums overflow anyway is
// queued for the exact CUDA-core fallback.
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
constexpr int kPanelBytesK = kTileKeys * 128;      // 256 keys x 64 bf16 = 32 KB
constexpr int kPanelBytesQ = kRowsPerTile * 128;   // 128 rows x 64 bf16 = 16 KB
constexpr uint32_t kTmemCols = 512;
constexpr long long kWaitLimit = 4000000000LL;     // cycles, ~2 s

template <int D>
struct Cfg {
    static constexpr int kPanels = D / 64;
    static constexpr int kQBytes = kPanels * kPanelBytesQ;
    static constexpr int kStages = D == 64 ? 5 : (D == 128 ? 4 : 3);
    static constexpr int kSmem = 2 * kQBytes + kStages * kPanelBytesK + 1024;
};

struct Shared {
    uint64_t kfull[8], kempty[8];
    uint64_t qfull[2], qempty[2];
    uint64_t tfull[2], tempty[2];
    uint64_t fin;
    uint32_t tmem_base;
    int abort;
};

struct Unit {
    SeqInfo sq;
    int j, mt, c, k0, k1, ntiles;
};

__device__ __forceinline__ void decode_unit(const ScoreParams &p, int u, Unit &un) {
    const int s = find_seq_by_unit(p.seqs, p.num_seqs, u);
    un.sq = p.seqs[s];
    int loc = u - un.sq.unit_off;
    un.mt = loc % un.sq.mtiles;
    loc /= un.sq.mtiles;
    un.c = loc % un.sq.nchunks;
    un.j = loc / un.sq.nchunks;
    un.k0 = un.c * p.C;
    un.k1 = min(un.k0 + p.C, un.sq.L);
    un.ntiles = (un.k1 - un.k0 + kTileKeys - 1) / kTileKeys;
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
        for (int t = 0; t < un.ntiles; ++t) {
            const int row0 = un.sq.tok_off + un.k0 + t * kTileKeys;
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
    constexpr int kTotal = kRowsPerTile * kCh;
    constexpr int kBatch = 8;
    volatile int *abort = &sh.abort;
    const int qt = threadIdx.x - kWarpQ * 32;
    uint32_t ui = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++ui) {
        Unit un;
        decode_unit(p, u, un);
        const int qb = ui & 1;
        if (!mbar_wait(smem_u32(&sh.qempty[qb]), ((ui >> 1) & 1) ^ 1, abort, kWaitLimit)) return;
        uint8_t *dst = qbuf + qb * C::kQBytes;
        const int ns = un.sq.ns;
        const int grows = p.g * ns;
        for (int base = qt; base < kTotal; base += kQThreads * kBatch) {
            uint4 v[kBatch];
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                const int idx = base + i * kQThreads;
                v[i] = make_uint4(0, 0, 0, 0);
                if (idx < kTotal) {
                    const int row = idx / kCh, ch = idx % kCh;
                    const int rr = un.mt * kRowsPerTile + row;
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
                    const int pn = ch >> 3, c16 = ch & 7;
                    uint8_t *d = dst + pn * kPanelBytesQ + row * 128 + ((c16 ^ (row & 7)) << 4);
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
    constexpr uint32_t idesc = idesc_bf16_f32(kRowsPerTile, kTileKeys);
    volatile int *abort = &sh.abort;
    uint32_t it = 0, tile = 0, ui = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++ui) {
        Unit un;
        decode_unit(p, u, un);
        const int qb = ui & 1;
        if (!mbar_wait(smem_u32(&sh.qfull[qb]), (ui >> 1) & 1, abort, kWaitLimit)) goto out;
        tc_fence_after();
        {
            const uint32_t qaddr = smem_u32(qbuf + qb * C::kQBytes);
            for (int t = 0; t < un.ntiles; ++t, ++tile) {
                const int b = tile & 1;
                if (!mbar_wait(smem_u32(&sh.tempty[b]), ((tile >> 1) & 1) ^ 1, abort, kWaitLimit))
                    goto out;
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(b * kTileKeys);
                for (int pn = 0; pn < C::kPanels; ++pn, ++it) {
                    const int st = it % C::kStages;
                    if (!mbar_wait(smem_u32(&sh.kfull[st]), (it / C::kStages) & 1, abort, kWaitLimit))
                        goto out;
                    tc_fence_after();
                    const uint64_t ad = smem_desc_sw128(qaddr + pn * kPanelBytesQ);
                    const uint64_t bd = smem_desc_sw128(smem_u32(kbuf + st * kPanelBytesK));
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)  // 4 x K=16 per 64-wide panel (32 bytes each)
                        mma_bf16(d_tmem, ad + 2 * ks, bd + 2 * ks, idesc, (pn | ks) != 0);
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

__device__ __forceinline__ float sum16(const float (&v)[32], int o) {
    const float a0 = (v[o + 0] + v[o + 1]) + (v[o + 2] + v[o + 3]);
    const float a1 = (v[o + 4] + v[o + 5]) + (v[o + 6] + v[o + 7]);
    const float a2 = (v[o + 8] + v[o + 9]) + (v[o + 10] + v[o + 11]);
    const float a3 = (v[o + 12] + v[o + 13]) + (v[o + 14] + v[o + 15]);
    return (a0 + a1) + (a2 + a3);
}

template <int D, int G>
__device__ void role_softmax(const ScoreParams &p, Shared &sh, uint32_t tmem, int units) {
    volatile int *abort = &sh.abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wg = (warp - kWarpEpi) >> 2;  // warpgroup: TMEM buffer and tile parity
    const int quarter = warp & 3;           // TMEM lanes 32*quarter .. +31
    const int row = quarter * 32 + lane;
    const float s = p.scale_log2;
    uint32_t tile = 0, mine = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        Unit un;
        decode_unit(p, u, un);
        const SeqInfo &sq = un.sq;
        const int grows = p.g * sq.ns;
        const int rl = un.mt * kRowsPerTile + row;
        const bool valid = rl < grows;
        const int a = sq.L - sq.ns + (valid ? rl % sq.ns : 0);  // causal limit of this row
        const int64_t r = (int64_t)un.j * grows + rl;           // h * n_s + t
        float *part = p.part + sq.part_off + r;
        const int par = (wg ^ (int)(tile & 1)) & 1;  // which tiles of the unit are ours
        float ref = -INFINITY, bias = 0.f, lsum = 0.f;
        bool have_ref = false;
        for (int tt = par; tt < un.ntiles; tt += 2) {
            const bool ok = mbar_wait(smem_u32(&sh.tfull[wg]), mine & 1, abort, kWaitLimit);
            __syncwarp();  // tcgen05.ld is warp-collective: reconverge after polling
            if (!__all_sync(0xffffffffu, ok)) return;
            tc_fence_after();
            const uint32_t taddr =
                tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(wg * kTileKeys);
            const int key0 = un.k0 + tt * kTileKeys;
            const bool masked = key0 + kTileKeys - 1 > sq.L - sq.ns;
            if (!have_ref) {
                float mx = -INFINITY;
#pragma unroll 1
                for (int cg = 0; cg < kTileKeys / 32; ++cg) {
                    float v[32];
                    tmem_ld32(taddr + cg * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float x = (masked && key0 + cg * 32 + i > a) ? -INFINITY : v[i];
                        mx = fmaxf(mx, x);
                    }
                }
                ref = mx * s;
                bias = (ref == -INFINITY) ? -INFINITY : -ref;
                have_ref = true;
            }
            float acc = 0.f;
#pragma unroll
            for (int cg = 0; cg < kTileKeys / 32; ++cg) {
                float v[32];
                tmem_ld32(taddr + cg * 32, v);
                tmem_wait_ld();
                if (masked) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = (key0 + cg * 32 + i > a) ? -INFINITY : v[i];
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = ex2_approx(fmaf(v[i], s, bias));
                const float lo = sum16(v, 0), hi = sum16(v, 16);
                const int kb = key0 + cg * 32;
                if constexpr (G == 16) {
                    const int b = kb / 16;
                    if (valid && b < sq.nb) part[(int64_t)b * sq.R] = lo;
                    if (valid && b + 1 < sq.nb) part[(int64_t)(b + 1) * sq.R] = hi;
                    lsum += lo;
                    lsum += hi;
                } else if constexpr (G == 32) {
                    const float bs = lo + hi;
                    const int b = kb / 32;
                    if (valid && b < sq.nb) part[(int64_t)b * sq.R] = bs;
                    lsum += bs;
                } else {
                    acc += lo + hi;
                    if ((cg + 1) % (G / 32) == 0) {
                        const int b = (kb + 32 - G) / G;
                        if (valid && b < sq.nb) part[(int64_t)b * sq.R] = acc;
                        lsum += acc;
                        acc = 0.f;
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&sh.tempty[wg]));
            ++mine;
        }
        if (valid) {
            const int64_t o = sq.stat_off + (int64_t)(kSlotsPerChunk * un.c + par) * sq.R + r;
            p.mref[o] = ref;
            p.lsum[o] = lsum;
        }
        // fp32 overflow of the sums (logits far above this warpgroup's reference):
        // queue the unit for the exact fallback
        const bool bad = valid && !(lsum <= 3.0e38f);
        if (__any_sync(0xffffffffu, bad) && lane == 0) {
            const int idx = atomicAdd(&const_cast<Counters *>(p.counters)->flagged, 1);
            if (idx < p.flag_cap) p.flag_list[idx] = u;
        }
        tile += un.ntiles;
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
    uint8_t *qbuf = smem;                    // 2 x Q tile (1024-aligned panels)
    uint8_t *kbuf = smem + 2 * C::kQBytes;   // kStages x K panel
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
            mbar_init(smem_u32(&sh.tempty[b]), kEpiThreads);
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

// K viewed as a 2-D row-major matrix [total_tokens, Hk*d]; one box = 256 rows
// (keys) x 64 columns (head dims) with the 128-byte swizzle.  Rows past the end
// read as zeros.
bool encode_k_map(CUtensorMap *tm, const ScoreParams &p, int64_t total_tokens) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)p.Hk * p.d, (cuuint64_t)total_tokens};
    const cuuint64_t strides[1] = {(cuuint64_t)p.Hk * p.d * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kTileKeys};
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
