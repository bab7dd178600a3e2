// api.cu -- the C ABI declared in include/up.h: argument validation, workspace
// layout, per-device state and kernel launches.  No compute happens here.
#include <atomic>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "../../include/up.h"
#include "common.cuh"

namespace {

// A named NVTX range around each public call's host work (argument checks and
// launches), so a timeline profiler shows the three calls of a step; without
// a profiler attached a push or pop is a check of a null hook.
struct CallRange {
    explicit CallRange(const char *name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
    CallRange(const CallRange &) = delete;
    CallRange &operator=(const CallRange &) = delete;
};

// Sticky device error word (UP_DEVERR_* bits), one per device.
__device__ unsigned int g_up_device_error;

struct DeviceState {
    bool ready = false;
    int sms = 0;
    unsigned int *err = nullptr;
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// optional events recorded around the tensor-core scoring kernel (per host thread)
thread_local cudaEvent_t t_kernel_start = nullptr, t_kernel_stop = nullptr;

// Bound of the scoring kernel's spin-waits in SM clock cycles (about two
// seconds at the GB300's clocks unless a test lowers it).
constexpr long long kDefaultWaitLimit = 4000000000LL;
std::atomic<long long> g_wait_limit{kDefaultWaitLimit};

up_status device_state(DeviceState **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return UP_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return UP_ERR_CUDA;
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_up_device_error) != cudaSuccess) return UP_ERR_CUDA;
        d.err = static_cast<unsigned int *>(p);
        d.ready = true;
    }
    *out = &d;
    return UP_OK;
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace

namespace up {
unsigned int *device_error_word() {
    DeviceState *ds = nullptr;
    return device_state(&ds) == UP_OK ? ds->err : nullptr;
}
}  // namespace up

namespace {

bool valid_G(int G) { return G == 16 || G == 32 || G == 64 || G == 128 || G == 256; }
bool valid_d(int d) { return d == 64 || d == 128 || d == 256; }
bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Keys per work unit (a multiple of 256).  The CTAs of the score kernel walk
// the units round-robin, so the step count of the slowest CTA is
// ceil(units / CTAs) * C; C is chosen to minimise that, plus a per-unit cost of
// refilling the Q tiles (about 256 keys' worth), over C in 256..16384.  A function
// of the call's shape and the device's SM count only, so scores are
// reproducible on a given GPU model.
constexpr int kMaxChunk = 16384;

int choose_chunk(int B, int64_t total, int Hq, int Hk, int d, int n, int ctas) {
    const int g = Hq / Hk;
    const int64_t nn = n < total ? n : total;
    const int64_t tpt = up::tokens_per_tile(g), tpu = up::tiles_per_unit(d);
    const int64_t groups = (int64_t)Hk * (((nn + tpt - 1) / tpt + tpu - 1) / tpu);
    int best = up::kChunkQuantum;
    int64_t best_cost = INT64_MAX;
    for (int C = up::kChunkQuantum; C <= kMaxChunk; C += up::kChunkQuantum) {
        const int64_t units = groups * ((total + C - 1) / C + (B > 1 ? B - 1 : 0));
        const int64_t waves = (units + ctas - 1) / (ctas > 0 ? ctas : 1);
        const int64_t cost = waves * (C + 256);
        if (cost < best_cost) { best_cost = cost; best = C; }
    }
    return best;
}

// Workspace layout for a given chunk size.  The smallest chunk needs the most
// statistics, so sizing the workspace with C = 256 covers every chunk choice.
up::ScoreLayout score_layout(int B, int64_t total, int Hq, int Hk, int d, int n, int G, int chunk) {
    up::ScoreLayout L{};
    const int g = Hq / Hk;
    L.total_tokens = total;
    L.chunk = chunk;
    const int64_t nn = n < total ? n : total;
    const int64_t ns_sum = ((int64_t)n * B < total) ? (int64_t)n * B : total;
    L.max_blocks = total / G + B;
    L.max_rows = (int64_t)Hq * ns_sum;
    L.max_part = (int64_t)Hq * nn * L.max_blocks;
    const int64_t max_chunks = total / L.chunk + B;
    L.max_stat = (int64_t)Hq * nn * max_chunks * up::kSlotsPerChunk;
    const int64_t tpt = up::tokens_per_tile(g), tpu = up::tiles_per_unit(d);
    L.max_units = (int64_t)Hk * (((nn + tpt - 1) / tpt + tpu - 1) / tpu) * max_chunks;
    L.max_qrows = ns_sum;
    size_t off = 0;
    L.seqs = off;     off = align256(off + sizeof(up::SeqInfo) * (size_t)(B > 0 ? B : 1));
    L.counters = off; off = align256(off + sizeof(up::Counters));
    L.part = off;     off = align256(off + sizeof(float) * (size_t)L.max_part);
    L.mref = off;     off = align256(off + sizeof(float) * (size_t)L.max_stat);
    L.lsum = off;     off = align256(off + sizeof(float) * (size_t)L.max_stat);
    L.flags = off;    off = align256(off + sizeof(int32_t) * (size_t)(32 * L.max_units + 16));
    L.total = off;
    return L;
}

struct CompactLayout {
    size_t nkept, list, dst_blk, total;
};

CompactLayout compact_layout(int B, int64_t total, int G) {
    CompactLayout L{};
    const int64_t max_blocks = total / G + B;
    size_t off = 0;
    L.nkept = off;   off = align256(off + 256);
    L.list = off;    off = align256(off + sizeof(int4) * (size_t)(max_blocks > 0 ? max_blocks : 1));
    L.dst_blk = off; off = align256(off + sizeof(int32_t) * (size_t)(max_blocks > 0 ? max_blocks : 1));
    L.total = off;
    return L;
}

}  // namespace

extern "C" {

const char *up_status_string(up_status status) {
    switch (status) {
        case UP_OK: return "ok";
        case UP_ERR_INVALID_ARG: return "invalid argument";
        case UP_ERR_UNSUPPORTED: return "unsupported configuration";
        case UP_ERR_WORKSPACE: return "workspace missing or too small";
        case UP_ERR_CUDA: return "CUDA error";
        case UP_ERR_TIMEOUT: return "device-side bounded wait expired";
        case UP_ERR_DEVICE: return "device-side argument check failed";
    }
    return "unknown status";
}

up_status up_set_kernel_timing_events(up_event_t start_event, up_event_t stop_event) {
    if ((start_event == nullptr) != (stop_event == nullptr)) return UP_ERR_INVALID_ARG;
    t_kernel_start = reinterpret_cast<cudaEvent_t>(start_event);
    t_kernel_stop = reinterpret_cast<cudaEvent_t>(stop_event);
    return UP_OK;
}

up_status up_set_wait_limit(uint64_t cycles) {
    if (cycles > (uint64_t)kDefaultWaitLimit) return UP_ERR_INVALID_ARG;
    g_wait_limit.store(cycles == 0 ? kDefaultWaitLimit : (long long)cycles);
    return UP_OK;
}

up_status up_get_device_error(uint32_t *bits) {
    if (!bits) return UP_ERR_INVALID_ARG;
    DeviceState *ds = nullptr;
    up_status st = device_state(&ds);
    if (st != UP_OK) return st;
    unsigned int v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return UP_ERR_CUDA;
    if (cudaMemcpy(&v, ds->err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return UP_ERR_CUDA;
    if (cudaMemset(ds->err, 0, sizeof v) != cudaSuccess) return UP_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return UP_ERR_CUDA;
    *bits = v;
    if (v & UP_DEVERR_TIMEOUT) return UP_ERR_TIMEOUT;
    return v ? UP_ERR_DEVICE : UP_OK;
}

}  // extern "C"

namespace {

up_status check_score_args(const void *q_last, const void *k, const int32_t *cu_seqlens,
                           int num_seqs, int64_t total_tokens, int Hq, int Hk, int d, int n,
                           int G, const float *scores, const int32_t *cu_blocks) {
    if (num_seqs < 0 || total_tokens < 0 || total_tokens > INT32_MAX) return UP_ERR_INVALID_ARG;
    if (!cu_seqlens || !cu_blocks) return UP_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q_last || !k || !scores)) return UP_ERR_INVALID_ARG;
    if (Hq < 1 || Hk < 1 || Hq % Hk != 0 || n < 1 || d < 1 || G < 1) return UP_ERR_INVALID_ARG;
    if (Hq / Hk > 16 || !valid_d(d) || !valid_G(G) || n > 1024) return UP_ERR_UNSUPPORTED;
    if (!aligned(q_last, 16) || !aligned(k, 16) || !aligned(scores, 4)) return UP_ERR_INVALID_ARG;
    return UP_OK;
}

// Keys in a paged cache (see up_score_blocks_paged); block_table == nullptr:
// token-major keys.
struct PagedKeys {
    const int32_t *block_table;
    int page_size, max_pages;
    int64_t num_pages;
};

// The scoring call: plan, then the tensor-core kernel (scores included).  Hq_norm is
// the head count the mean over heads divides by (Hq, or all tensor-parallel
// ranks' heads); pk describes paged keys (none: token-major k).
up_status score_impl(const void *q_last, const void *k, const int32_t *cu_seqlens,
                     int num_seqs, int64_t total_tokens, int Hq, int Hk, int d, int n, int G,
                     int Hq_norm, const PagedKeys &pk, float *scores, int32_t *cu_blocks,
                     void *workspace, size_t workspace_bytes, up_stream_t stream) {
    up_status st = check_score_args(q_last, k, cu_seqlens, num_seqs, total_tokens, Hq, Hk, d, n,
                                    G, scores, cu_blocks);
    if (st != UP_OK) return st;
    if (!workspace || !aligned(workspace, 256) ||
        workspace_bytes < score_layout(num_seqs, total_tokens, Hq, Hk, d, n, G, up::kChunkQuantum).total)
        return UP_ERR_WORKSPACE;
    DeviceState *ds = nullptr;
    if ((st = device_state(&ds)) != UP_OK) return st;
    const int chunk = choose_chunk(num_seqs, total_tokens, Hq, Hk, d, n, ds->sms);
    const up::ScoreLayout lay = score_layout(num_seqs, total_tokens, Hq, Hk, d, n, G, chunk);
    if (workspace_bytes < lay.total) return UP_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    up::ScoreParams p{};
    p.q = static_cast<const __nv_bfloat16 *>(q_last);
    p.k = static_cast<const __nv_bfloat16 *>(k);
    p.seqs = reinterpret_cast<const up::SeqInfo *>(ws + lay.seqs);
    p.counters = reinterpret_cast<const up::Counters *>(ws + lay.counters);
    p.part = reinterpret_cast<float *>(ws + lay.part);
    p.mref = reinterpret_cast<float *>(ws + lay.mref);
    p.lsum = reinterpret_cast<float *>(ws + lay.lsum);
    p.scores = scores;
    p.flag_list = reinterpret_cast<int32_t *>(ws + lay.flags);
    p.max_units = (int)lay.max_units;
    p.flag_cap = (int)(32 * lay.max_units + 16);
    p.num_seqs = num_seqs;
    p.Hq = Hq; p.Hk = Hk; p.g = Hq / Hk; p.d = d; p.n = n; p.G = G; p.C = lay.chunk;
    p.Hq_norm = Hq_norm;
    p.block_table = pk.block_table;
    p.page_size = pk.page_size;
    p.max_pages = pk.max_pages;
    p.num_pages = pk.num_pages;
    p.tpt = up::tokens_per_tile(p.g);
    p.scale_log2 = (float)(1.4426950408889634 / __builtin_sqrt((double)d));
    p.wait_limit = g_wait_limit.load();
    p.err = ds->err;
    p.part_cap = lay.max_part;
    p.stat_cap = lay.max_stat;
    p.scores_cap = lay.max_blocks;
    p.cu_seqlens = cu_seqlens;
    if (num_seqs == 1) {  // the plan's row for the only sequence, from the host's sizes
        const int64_t L = total_tokens, ns = L < n ? L : n;
        const int64_t tpt = up::tokens_per_tile(p.g), tpu = up::tiles_per_unit(d);
        up::SeqInfo &si = p.seq0;
        si = up::SeqInfo{};
        si.L = (int32_t)L;
        si.ns = (int32_t)ns;
        si.nb = (int32_t)((L + G - 1) / G);
        si.nchunks = (int32_t)((L + p.C - 1) / p.C);
        si.mtiles = (int32_t)(((ns + tpt - 1) / tpt + tpu - 1) / tpu);
        si.R = (int32_t)(Hq * ns);
        p.units0 = Hk * si.mtiles * si.nchunks;
    }
    if (up::launch_score_plan(cu_seqlens, cu_blocks, p, total_tokens, s) != cudaSuccess)
        return UP_ERR_CUDA;
    if (num_seqs == 0 || total_tokens == 0) return UP_OK;
    if (t_kernel_start && cudaEventRecord(t_kernel_start, s) != cudaSuccess) return UP_ERR_CUDA;
    if (up::launch_score_main(p, lay, ds->sms, s) != cudaSuccess) return UP_ERR_CUDA;
    if (t_kernel_stop && cudaEventRecord(t_kernel_stop, s) != cudaSuccess) return UP_ERR_CUDA;
    return UP_OK;
}

}  // namespace

extern "C" {

size_t up_score_blocks_workspace(int num_seqs, int64_t total_tokens, int Hq, int Hk, int d,
                                 int n, int G) {
    if (check_score_args(reinterpret_cast<const void *>(16), reinterpret_cast<const void *>(16),
                         reinterpret_cast<const int32_t *>(16), num_seqs, total_tokens, Hq, Hk,
                         d, n, G, reinterpret_cast<const float *>(16),
                         reinterpret_cast<const int32_t *>(16)) != UP_OK)
        return 0;
    return score_layout(num_seqs, total_tokens, Hq, Hk, d, n, G, up::kChunkQuantum).total;
}

up_status up_score_blocks(const void *q_last, const void *k, const int32_t *cu_seqlens,
                          int num_seqs, int64_t total_tokens, int Hq, int Hk, int d, int n,
                          int G, float *scores, int32_t *cu_blocks, void *workspace,
                          size_t workspace_bytes, up_stream_t stream) {
    const CallRange range("up_score_blocks");
    return score_impl(q_last, k, cu_seqlens, num_seqs, total_tokens, Hq, Hk, d, n, G, Hq,
                      PagedKeys{}, scores, cu_blocks, workspace, workspace_bytes, stream);
}

up_status up_score_blocks_shard(const void *q_last, const void *k, const int32_t *cu_seqlens,
                                int num_seqs, int64_t total_tokens, int Hq, int Hk, int d, int n,
                                int G, int Hq_total, float *scores, int32_t *cu_blocks,
                                void *workspace, size_t workspace_bytes, up_stream_t stream) {
    const CallRange range("up_score_blocks_shard");
    if (Hq_total < Hq || Hq_total < 1) return UP_ERR_INVALID_ARG;
    return score_impl(q_last, k, cu_seqlens, num_seqs, total_tokens, Hq, Hk, d, n, G, Hq_total,
                      PagedKeys{}, scores, cu_blocks, workspace, workspace_bytes, stream);
}

up_status up_score_blocks_paged(const void *q_last, const void *k_pages, int64_t num_pages,
                                int page_size, const int32_t *block_table, int max_pages,
                                const int32_t *cu_seqlens, int num_seqs, int64_t total_tokens,
                                int Hq, int Hk, int d, int n, int G, float *scores,
                                int32_t *cu_blocks, void *workspace, size_t workspace_bytes,
                                up_stream_t stream) {
    const CallRange range("up_score_blocks_paged");
    if (!block_table || page_size < 128 || page_size % 128 != 0 || num_pages < 1 ||
        max_pages < 1 || Hk < 1 || num_pages * (int64_t)Hk * page_size >= ((int64_t)1 << 31))
        return UP_ERR_INVALID_ARG;
    // one sequence starts without the plan's checks: its table row must hold
    // total_tokens keys (the only valid length)
    if (num_seqs == 1 && (total_tokens + page_size - 1) / page_size > max_pages)
        return UP_ERR_INVALID_ARG;
    const PagedKeys pk{block_table, page_size, max_pages, num_pages};
    return score_impl(q_last, k_pages, cu_seqlens, num_seqs, total_tokens, Hq, Hk, d, n, G, Hq,
                      pk, scores, cu_blocks, workspace, workspace_bytes, stream);
}

up_status up_select_topp(const float *scores, const int32_t *cu_blocks,
                         const int32_t *cu_seqlens, int num_seqs, int G, double p,
                         uint8_t *keep, int32_t *kept_tokens, up_stream_t stream) {
    const CallRange range("up_select_topp");
    if (num_seqs < 0 || G < 1 || !(p > 0.0)) return UP_ERR_INVALID_ARG;
    if (!valid_G(G)) return UP_ERR_UNSUPPORTED;
    if (num_seqs > 0 && (!scores || !cu_blocks || !cu_seqlens || !keep || !kept_tokens))
        return UP_ERR_INVALID_ARG;
    DeviceState *ds = nullptr;
    up_status st = device_state(&ds);
    if (st != UP_OK) return st;
    if (up::launch_select(scores, cu_blocks, cu_seqlens, num_seqs, G, false, p, 0, false, keep,
                          kept_tokens, ds->err, ds->sms, reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return UP_ERR_CUDA;
    return UP_OK;
}

up_status up_select_blocks(const float *scores, const int32_t *cu_blocks,
                           const int32_t *cu_seqlens, int num_seqs, int G, up_select_mode mode,
                           double p, int k, uint32_t flags, uint8_t *keep, int32_t *kept_tokens,
                           up_stream_t stream) {
    const CallRange range("up_select_blocks");
    if (num_seqs < 0 || G < 1 || (flags & ~UP_SELECT_KEEP_LAST) != 0) return UP_ERR_INVALID_ARG;
    if (mode == UP_SELECT_TOP_P) {
        if (!(p > 0.0)) return UP_ERR_INVALID_ARG;
    } else if (mode == UP_SELECT_TOP_K) {
        if (k < 1) return UP_ERR_INVALID_ARG;
    } else {
        return UP_ERR_INVALID_ARG;
    }
    if (!valid_G(G)) return UP_ERR_UNSUPPORTED;
    if (num_seqs > 0 && (!scores || !cu_blocks || !cu_seqlens || !keep || !kept_tokens))
        return UP_ERR_INVALID_ARG;
    DeviceState *ds = nullptr;
    up_status st = device_state(&ds);
    if (st != UP_OK) return st;
    if (up::launch_select(scores, cu_blocks, cu_seqlens, num_seqs, G, mode == UP_SELECT_TOP_K, p,
                          k, (flags & UP_SELECT_KEEP_LAST) != 0, keep, kept_tokens, ds->err, ds->sms,
                          reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return UP_ERR_CUDA;
    return UP_OK;
}

up_status up_block_csr(const uint8_t *keep, const int32_t *cu_blocks, int num_seqs,
                       int32_t *indptr, int32_t *indices, up_stream_t stream) {
    const CallRange range("up_block_csr");
    if (num_seqs < 0 || !keep || !cu_blocks || !indptr || !indices) return UP_ERR_INVALID_ARG;
    DeviceState *ds = nullptr;
    up_status st = device_state(&ds);
    if (st != UP_OK) return st;
    if (up::launch_block_csr(keep, cu_blocks, num_seqs, indptr, indices,
                             reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return UP_ERR_CUDA;
    return UP_OK;
}

size_t up_compact_workspace(int num_seqs, int64_t total_tokens, int G) {
    if (num_seqs < 0 || total_tokens < 0 || total_tokens > INT32_MAX || !valid_G(G)) return 0;
    return compact_layout(num_seqs, total_tokens, G).total;
}

up_status up_compact(const void *x, const int32_t *pos, int hidden, const int32_t *cu_seqlens,
                     int num_seqs, int64_t total_tokens, int G, const uint8_t *keep,
                     const int32_t *cu_blocks, void *x_out, int32_t *pos_out,
                     int32_t *cu_seqlens_out, int32_t *src_idx, int32_t *total_kept,
                     void *workspace, size_t workspace_bytes, up_stream_t stream) {
    const CallRange range("up_compact");
    if (num_seqs < 0 || total_tokens < 0 || total_tokens > INT32_MAX || hidden < 1 || G < 1)
        return UP_ERR_INVALID_ARG;
    if (!valid_G(G)) return UP_ERR_UNSUPPORTED;
    if (hidden % 8 != 0) return UP_ERR_UNSUPPORTED;
    if (!cu_seqlens || !cu_blocks || !cu_seqlens_out || !total_kept) return UP_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!x || !pos || !keep || !x_out || !pos_out)) return UP_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(x_out, 16)) return UP_ERR_INVALID_ARG;
    const CompactLayout lay = compact_layout(num_seqs, total_tokens, G);
    if (!workspace || workspace_bytes < lay.total || !aligned(workspace, 256))
        return UP_ERR_WORKSPACE;
    DeviceState *ds = nullptr;
    up_status st = device_state(&ds);
    if (st != UP_OK) return st;
    char *ws = static_cast<char *>(workspace);
    up::CompactArgs a{};
    a.x = static_cast<const uint4 *>(x);
    a.pos = pos;
    a.cu_seqlens = cu_seqlens;
    a.keep = keep;
    a.cu_blocks = cu_blocks;
    a.x_out = static_cast<uint4 *>(x_out);
    a.pos_out = pos_out;
    a.cu_out = cu_seqlens_out;
    a.src_idx = src_idx;
    a.total_kept = total_kept;
    a.nkept = reinterpret_cast<int32_t *>(ws + lay.nkept);
    a.list = reinterpret_cast<int4 *>(ws + lay.list);
    a.dst_blk = reinterpret_cast<int32_t *>(ws + lay.dst_blk);
    a.err = ds->err;
    a.max_blocks = total_tokens / G + num_seqs;
    a.total_tokens = total_tokens;
    a.nb_one = num_seqs == 1 ? (int)((total_tokens + G - 1) / G) : -1;
    a.num_seqs = num_seqs;
    a.G = G;
    a.hidden = hidden;
    a.vec_per_row = (int64_t)hidden * 2 / 16;
    int rpi = (int)(32768 / ((int64_t)hidden * 2));
    if (rpi < 1) rpi = 1;
    if (rpi > G) rpi = G;
    a.rows_per_item = rpi;
    a.items_per_block = (G + rpi - 1) / rpi;
    if (up::launch_compact(a, ds->sms, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return UP_ERR_CUDA;
    return UP_OK;
}

}  // extern "C"
