// compact_noalloc.cu -- up_compact_noalloc: compaction without a caller workspace.
//
// Some callers cannot allocate device memory at the point where they compact:
// an inference engine that reserves nearly all HBM for its KV cache at start-up
// and has nothing left to hand out, or a latency-critical serving loop that
// must not call cudaMalloc (which can synchronise the whole device and stall
// every other stream).  For them this entry point runs the same two compaction
// kernels as up_compact, but takes its scratch (the kept-block list, the
// destination row of every block and the kept-block counter) from a fixed
// array compiled into the library instead of from a workspace argument.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// code holds it (about 1.3 MB) until the process exits.  Host code cannot use
// the array's name as a device address, so the first call on each device looks
// the address up with cudaGetSymbolAddress while that device is current.
// Batches of at most kCompactOneKernelBlocks possible blocks take the
// one-kernel compaction, which needs no scratch at all; larger ones (up to
// UP_COMPACT_NOALLOC_MAX_BLOCKS) use the array.
#include <mutex>

#include "../../include/up.h"
#include "common.cuh"

namespace {

constexpr int64_t kMaxBlocks = UP_COMPACT_NOALLOC_MAX_BLOCKS;
constexpr size_t kCounterBytes = 256;
constexpr size_t kListBytes = sizeof(int4) * (size_t)kMaxBlocks;
constexpr size_t kDstBytes = sizeof(int32_t) * (size_t)kMaxBlocks;
constexpr size_t kScratchBytes = kCounterBytes + kListBytes + kDstBytes;

// Shared by every call on a device; each call overwrites what it reads (the
// counter, the list entries it counts and the destination of every block), so
// nothing has to be cleared between calls.
static __device__ __align__(256) unsigned char g_compact_scratch[kScratchBytes];

struct NoAllocDevice {
    bool ready = false;
    int sms = 0;
    unsigned char *scratch = nullptr;  // device address of g_compact_scratch
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
NoAllocDevice g_devs[kMaxDevices];

up_status noalloc_setup(NoAllocDevice **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return UP_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    NoAllocDevice &d = g_devs[dev];
    if (!d.ready) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_compact_scratch) != cudaSuccess || p == nullptr)
            return UP_ERR_CUDA;
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return UP_ERR_CUDA;
        d.scratch = static_cast<unsigned char *>(p);
        d.ready = true;
    }
    *out = &d;
    return UP_OK;
}

bool is_block_size(int G) { return G == 16 || G == 32 || G == 64 || G == 128 || G == 256; }
bool is_aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" up_status up_compact_noalloc(const void *x, const int32_t *pos, int hidden,
                                        const int32_t *cu_seqlens, int num_seqs,
                                        int64_t total_tokens, int G, const uint8_t *keep,
                                        const int32_t *cu_blocks, void *x_out, int32_t *pos_out,
                                        int32_t *cu_seqlens_out, int32_t *src_idx,
                                        int32_t *total_kept, up_stream_t stream) {
    if (num_seqs < 0 || total_tokens < 0 || total_tokens > INT32_MAX || hidden < 1 || G < 1)
        return UP_ERR_INVALID_ARG;
    if (!is_block_size(G) || hidden % 8 != 0) return UP_ERR_UNSUPPORTED;
    if (!cu_seqlens || !cu_blocks || !cu_seqlens_out || !total_kept) return UP_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!x || !pos || !keep || !x_out || !pos_out)) return UP_ERR_INVALID_ARG;
    if (!is_aligned(x, 16) || !is_aligned(x_out, 16)) return UP_ERR_INVALID_ARG;
    // the largest block count this batch can have must fit the fixed scratch
    if (total_tokens / G + num_seqs > kMaxBlocks) return UP_ERR_WORKSPACE;
    NoAllocDevice *dev = nullptr;
    up_status st = noalloc_setup(&dev);
    if (st != UP_OK) return st;
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
    a.nkept = reinterpret_cast<int32_t *>(dev->scratch);
    a.list = reinterpret_cast<int4 *>(dev->scratch + kCounterBytes);
    a.dst_blk = reinterpret_cast<int32_t *>(dev->scratch + kCounterBytes + kListBytes);
    // the kernels check cu_blocks[num_seqs] against this bound on the device, so
    // a cu_blocks that disagrees with total_tokens never reaches past the array
    a.max_blocks = total_tokens / G + num_seqs;
    a.total_tokens = total_tokens;
    a.nb_one = num_seqs == 1 ? (int)((total_tokens + G - 1) / G) : -1;
    a.err = up::device_error_word();
    if (!a.err) return UP_ERR_CUDA;
    a.num_seqs = num_seqs;
    a.G = G;
    a.hidden = hidden;
    a.vec_per_row = (int64_t)hidden * 2 / 16;
    int rpi = (int)(32768 / ((int64_t)hidden * 2));
    if (rpi < 1) rpi = 1;
    if (rpi > G) rpi = G;
    a.rows_per_item = rpi;
    a.items_per_block = (G + rpi - 1) / rpi;
    if (up::launch_compact(a, dev->sms, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return UP_ERR_CUDA;
    return UP_OK;
}
