"""UniPrefill block-wise sparsification hot path for GB300 (sm_103a).

A thin ctypes binding over ``libup.so`` (see include/up.h): the functions here
check tensor dtypes/devices, allocate outputs with PyTorch and pass raw device
pointers and the current CUDA stream to the C ABI.  Every step of the path runs
in the library's CUDA kernels; there is no Python or CPU compute path.  If the
library is not built, every call raises.

    scores, cu_blocks = score_blocks(q_last, k, cu_seqlens, n, G)
    keep, kept_tokens = select_topp(scores, cu_blocks, cu_seqlens, G, p)
    x_out, pos_out, cu_out, total = compact(x, pos, cu_seqlens, G, keep, cu_blocks)
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

__all__ = ["build", "lib", "UpError", "score_blocks_workspace", "score_blocks",
           "score_blocks_paged", "block_csr", "shard_heads",
           "tp_score_blocks", "select_topp",
           "compact_workspace", "compact", "compact_noalloc", "set_kernel_timing_events",
           "set_wait_limit", "get_device_error", "Sparsifier", "SELECT_MAX_BLOCKS"]

SELECT_MAX_BLOCKS = 16384
_lib = None


class UpError(RuntimeError):
    def __init__(self, where, status):
        msg = lib().up_status_string(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")
        self.status = status


def build(force: bool = False) -> str:
    """Compile libup.so for sm_103a (nvcc) into the package's _build/ folder."""
    return _build.build(force=force)


def lib():
    """The loaded libup.so (ctypes).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        raise RuntimeError(f"{_build.LIB} is missing: build it with block_sparse_long_up_gb300.build()")
    _lib = load_library(_build.LIB)
    return _lib


def load_library(path):
    """Load a build of the C ABI at `path` (the library, or its checked
    variant from _build.build(checked=True)) with its ctypes signatures."""
    L = ctypes.CDLL(path)
    P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    L.up_status_string.argtypes = [I]
    L.up_status_string.restype = ctypes.c_char_p
    L.up_score_blocks_workspace.argtypes = [I, I64, I, I, I, I, I]
    L.up_score_blocks_workspace.restype = SZ
    L.up_score_blocks.argtypes = [P, P, P, I, I64, I, I, I, I, I, P, P, P, SZ, P]
    L.up_score_blocks.restype = I
    L.up_score_blocks_shard.argtypes = [P, P, P, I, I64, I, I, I, I, I, I, P, P, P, SZ, P]
    L.up_score_blocks_shard.restype = I
    L.up_score_blocks_paged.argtypes = [P, P, I64, I, P, I, P, I, I64, I, I, I, I, I, P, P, P,
                                        SZ, P]
    L.up_score_blocks_paged.restype = I
    L.up_block_csr.argtypes = [P, P, I, P, P, P]
    L.up_block_csr.restype = I
    L.up_select_topp.argtypes = [P, P, P, I, I, ctypes.c_double, P, P, P]
    L.up_select_topp.restype = I
    L.up_select_blocks.argtypes = [P, P, P, I, I, I, ctypes.c_double, I, ctypes.c_uint32, P, P, P]
    L.up_select_blocks.restype = I
    L.up_compact_workspace.argtypes = [I, I64, I]
    L.up_compact_workspace.restype = SZ
    L.up_compact.argtypes = [P, P, I, P, I, I64, I, P, P, P, P, P, P, P, P, SZ, P]
    L.up_compact.restype = I
    L.up_compact_noalloc.argtypes = [P, P, I, P, I, I64, I, P, P, P, P, P, P, P, P]
    L.up_compact_noalloc.restype = I
    L.up_set_kernel_timing_events.argtypes = [P, P]
    L.up_set_kernel_timing_events.restype = I
    L.up_get_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    L.up_get_device_error.restype = I
    L.up_measure_ex2_rate.argtypes = [ctypes.POINTER(ctypes.c_double), P]
    L.up_measure_ex2_rate.restype = I
    L.up_set_wait_limit.argtypes = [ctypes.c_uint64]
    L.up_set_wait_limit.restype = I
    return L


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _need_rows(t, name, dtype, device):
    """x or pos of a compaction: a CUDA tensor on `device`, or a pinned (page-
    locked) host tensor, which the kernel reads in place through unified
    addressing (only the kept rows cross the host link)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.is_cuda:
        _need(t, name, dtype, device)
        return
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not t.is_pinned():
        raise ValueError(f"{name} must be a CUDA tensor or a pinned host tensor")


def _check(where, status):
    if status != 0:
        raise UpError(where, status)


def _alloc_ws(nbytes, device):
    # 256-byte alignment comes with the caching allocator's blocks
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def score_blocks_workspace(num_seqs, total_tokens, Hq, Hk, d, n, G) -> int:
    return int(lib().up_score_blocks_workspace(num_seqs, total_tokens, Hq, Hk, d, n, G))


def score_blocks(q_last, k, cu_seqlens, n, G, scores=None, cu_blocks=None, workspace=None,
                 stream=None, Hq_total=None):
    """Block scores (fp32 [sum nb_s]) and cu_blocks (int32 [B+1]); see up_score_blocks.

    With Hq_total (the query heads of all tensor-parallel ranks), q_last and k
    hold one rank's heads and the mean over heads divides by Hq_total
    (up_score_blocks_shard): the shards' scores sum to the scores of all heads."""
    _need(k, "k", torch.bfloat16)
    dev = k.device
    _need(q_last, "q_last", torch.bfloat16, dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
    total, Hk, d = k.shape
    Hq = q_last.shape[1]
    B = cu_seqlens.numel() - 1
    cap = total // G + B
    if scores is None:
        scores = torch.empty(max(cap, 1), dtype=torch.float32, device=dev)
    if cu_blocks is None:
        cu_blocks = torch.empty(B + 1, dtype=torch.int32, device=dev)
    _need(scores, "scores", torch.float32, dev)
    _need(cu_blocks, "cu_blocks", torch.int32, dev)
    if scores.numel() < cap:
        raise ValueError(f"scores needs {cap} entries")
    ws_need = score_blocks_workspace(B, total, Hq, Hk, d, n, G)
    if workspace is None:
        workspace = _alloc_ws(ws_need, dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    if Hq_total is None:
        st = lib().up_score_blocks(_ptr(q_last), _ptr(k), _ptr(cu_seqlens), B, total, Hq, Hk, d,
                                   n, G, _ptr(scores), _ptr(cu_blocks), _ptr(workspace), ws_bytes,
                                   _stream(stream))
        _check("up_score_blocks", st)
    else:
        st = lib().up_score_blocks_shard(_ptr(q_last), _ptr(k), _ptr(cu_seqlens), B, total, Hq,
                                         Hk, d, n, G, int(Hq_total), _ptr(scores),
                                         _ptr(cu_blocks), _ptr(workspace), ws_bytes,
                                         _stream(stream))
        _check("up_score_blocks_shard", st)
    return scores, cu_blocks


def score_blocks_paged(q_last, k_pages, block_table, cu_seqlens, total_tokens, n, G,
                       scores=None, cu_blocks=None, workspace=None, stream=None):
    """Block scores with the keys in a paged cache (chunked prefill); see
    up_score_blocks_paged.  k_pages bf16 [num_pages, Hk, page_size, d];
    block_table int32 [num_seqs, max_pages] (key t of sequence s is row
    t % page_size of page block_table[s, t // page_size]); total_tokens = the
    sum of the sequence lengths (cu_seqlens[-1])."""
    _need(k_pages, "k_pages", torch.bfloat16)
    dev = k_pages.device
    _need(q_last, "q_last", torch.bfloat16, dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
    _need(block_table, "block_table", torch.int32, dev)
    num_pages, Hk, page_size, d = k_pages.shape
    Hq = q_last.shape[1]
    B = cu_seqlens.numel() - 1
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [num_seqs, max_pages]")
    total = int(total_tokens)
    cap = total // G + B
    if scores is None:
        scores = torch.empty(max(cap, 1), dtype=torch.float32, device=dev)
    if cu_blocks is None:
        cu_blocks = torch.empty(B + 1, dtype=torch.int32, device=dev)
    _need(scores, "scores", torch.float32, dev)
    _need(cu_blocks, "cu_blocks", torch.int32, dev)
    if scores.numel() < cap:
        raise ValueError(f"scores needs {cap} entries")
    if workspace is None:
        workspace = _alloc_ws(score_blocks_workspace(B, total, Hq, Hk, d, n, G), dev)
    st = lib().up_score_blocks_paged(_ptr(q_last), _ptr(k_pages), num_pages, page_size,
                                     _ptr(block_table), block_table.shape[1], _ptr(cu_seqlens), B,
                                     total, Hq, Hk, d, n, G, _ptr(scores), _ptr(cu_blocks),
                                     _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     _stream(stream))
    _check("up_score_blocks_paged", st)
    return scores, cu_blocks


def block_csr(keep, cu_blocks, indptr=None, indices=None, stream=None):
    """The kept blocks as a block-CSR matrix (indptr int32 [B+1], indices int32
    [sum nb_s] capacity; entries indptr[s]..indptr[s+1]-1 are sequence s's kept
    block numbers, ascending); see up_block_csr."""
    _need(keep, "keep", torch.uint8)
    dev = keep.device
    _need(cu_blocks, "cu_blocks", torch.int32, dev)
    B = cu_blocks.numel() - 1
    if indptr is None:
        indptr = torch.empty(B + 1, dtype=torch.int32, device=dev)
    if indices is None:
        indices = torch.empty(max(keep.numel(), 1), dtype=torch.int32, device=dev)
    _need(indptr, "indptr", torch.int32, dev)
    _need(indices, "indices", torch.int32, dev)
    _check("up_block_csr", lib().up_block_csr(_ptr(keep), _ptr(cu_blocks), B, _ptr(indptr),
                                               _ptr(indices), _stream(stream)))
    return indptr, indices


def shard_heads(q_last, k, rank, world):
    """This rank's tensor-parallel shard: KV heads [r*Hk/W, (r+1)*Hk/W) and the
    query heads of their GQA groups (views of q_last [rows, Hq, d] and k
    [tokens, Hk, d], made contiguous).  Hk must divide by the world size."""
    Hq, Hk = q_last.shape[1], k.shape[1]
    if Hk % world != 0:
        raise ValueError(f"{Hk} KV heads do not split over {world} ranks")
    hk = Hk // world
    g = Hq // Hk
    q = q_last[:, rank * hk * g:(rank + 1) * hk * g].contiguous()
    kk = k[:, rank * hk:(rank + 1) * hk].contiguous()
    return q, kk


def tp_score_blocks(q_last_shard, k_shard, cu_seqlens, n, G, Hq_total, group=None, stream=None):
    """Tensor-parallel block scores: this rank scores its head shard with the mean
    over all Hq_total query heads (up_score_blocks_shard), then a sum all-reduce
    over the process group gives every rank the scores of all heads (UniPrefill
    overview, fused-kernel paragraph).  Returns (scores, cu_blocks) as
    score_blocks; every rank then selects on identical scores.

    Everything (the zero fill, the scoring launches and the all-reduce) is
    issued on `stream` (default: the current stream), so the three are ordered
    on one stream whichever stream the caller passes."""
    import contextlib

    import torch.distributed as dist
    if k_shard.is_cuda:
        s = torch.cuda.current_stream(k_shard.device) if stream is None else stream
        on_stream = torch.cuda.stream(s)
    else:  # host tensors reach here only with a substituted score_blocks (CPU ranks)
        s, on_stream = stream, contextlib.nullcontext()
    with on_stream:
        # capacity past sum nb_s is summed too: start it at zero
        cap = k_shard.shape[0] // G + cu_seqlens.numel() - 1
        scores = torch.zeros(max(cap, 1), dtype=torch.float32, device=k_shard.device)
        scores, cu_blocks = score_blocks(q_last_shard, k_shard, cu_seqlens, n, G, scores=scores,
                                         stream=s, Hq_total=Hq_total)
        if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
            dist.all_reduce(scores, op=dist.ReduceOp.SUM, group=group)
    return scores, cu_blocks


def select_topp(scores, cu_blocks, cu_seqlens, G, p, keep=None, kept_tokens=None, stream=None):
    """Top-p keep flags (uint8 [sum nb_s]) and kept tokens per sequence (int32 [B])."""
    _need(scores, "scores", torch.float32)
    dev = scores.device
    _need(cu_blocks, "cu_blocks", torch.int32, dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
    B = cu_seqlens.numel() - 1
    if keep is None:
        keep = torch.empty(max(scores.numel(), 1), dtype=torch.uint8, device=dev)
    if kept_tokens is None:
        kept_tokens = torch.empty(max(B, 1), dtype=torch.int32, device=dev)
    _need(keep, "keep", torch.uint8, dev)
    _need(kept_tokens, "kept_tokens", torch.int32, dev)
    st = lib().up_select_topp(_ptr(scores), _ptr(cu_blocks), _ptr(cu_seqlens), B, G, float(p),
                              _ptr(keep), _ptr(kept_tokens), _stream(stream))
    _check("up_select_topp", st)
    return keep, kept_tokens


SELECT_MODES = {"top_p": 0, "top_k": 1}
SELECT_KEEP_LAST = 0x1


def select_blocks(scores, cu_blocks, cu_seqlens, G, mode="top_p", p=0.99, k=1, keep_last=False,
                  keep=None, kept_tokens=None, stream=None):
    """Block selection, general form: mode "top_p" (threshold p) or "top_k" (the
    first k ranks), optionally also keeping each sequence's last block.  Returns
    (keep uint8 [sum nb_s], kept_tokens int32 [B])."""
    if mode not in SELECT_MODES:
        raise ValueError(f"mode must be one of {sorted(SELECT_MODES)}")
    _need(scores, "scores", torch.float32)
    dev = scores.device
    _need(cu_blocks, "cu_blocks", torch.int32, dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
    B = cu_seqlens.numel() - 1
    if keep is None:
        keep = torch.empty(max(scores.numel(), 1), dtype=torch.uint8, device=dev)
    if kept_tokens is None:
        kept_tokens = torch.empty(max(B, 1), dtype=torch.int32, device=dev)
    _need(keep, "keep", torch.uint8, dev)
    _need(kept_tokens, "kept_tokens", torch.int32, dev)
    flags = SELECT_KEEP_LAST if keep_last else 0
    st = lib().up_select_blocks(_ptr(scores), _ptr(cu_blocks), _ptr(cu_seqlens), B, G,
                                SELECT_MODES[mode], float(p), int(k), flags, _ptr(keep),
                                _ptr(kept_tokens), _stream(stream))
    _check("up_select_blocks", st)
    return keep, kept_tokens


def compact_workspace(num_seqs, total_tokens, G) -> int:
    return int(lib().up_compact_workspace(num_seqs, total_tokens, G))


def compact(x, pos, cu_seqlens, G, keep, cu_blocks, x_out=None, pos_out=None,
            cu_seqlens_out=None, src_idx=None, total_kept=None, workspace=None, stream=None,
            want_src_idx=True):
    """Gather kept rows.  Outputs are sized for keeping everything; the true
    row count is total_kept (int32 [1], on the device).  x and pos may be
    pinned host tensors: the kernel then reads the kept rows in place."""
    _need(keep, "keep", torch.uint8)
    dev = keep.device
    _need_rows(x, "x", torch.bfloat16, dev)
    _need_rows(pos, "pos", torch.int32, dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
    _need(cu_blocks, "cu_blocks", torch.int32, dev)
    total, hidden = x.shape
    B = cu_seqlens.numel() - 1
    if x_out is None:
        x_out = torch.empty(max(total, 1), hidden, dtype=torch.bfloat16, device=dev)
    if pos_out is None:
        pos_out = torch.empty(max(total, 1), dtype=torch.int32, device=dev)
    if cu_seqlens_out is None:
        cu_seqlens_out = torch.empty(B + 1, dtype=torch.int32, device=dev)
    if src_idx is None and want_src_idx:
        src_idx = torch.empty(max(total, 1), dtype=torch.int32, device=dev)
    if total_kept is None:
        total_kept = torch.empty(1, dtype=torch.int32, device=dev)
    if x_out.shape[0] < total or pos_out.numel() < total:
        raise ValueError("x_out/pos_out must hold total_tokens rows")
    ws_need = compact_workspace(B, total, G)
    if workspace is None:
        workspace = _alloc_ws(ws_need, dev)
    st = lib().up_compact(_ptr(x), _ptr(pos), hidden, _ptr(cu_seqlens), B, total, G, _ptr(keep),
                          _ptr(cu_blocks), _ptr(x_out), _ptr(pos_out), _ptr(cu_seqlens_out),
                          _ptr(src_idx), _ptr(total_kept), _ptr(workspace),
                          workspace.numel() * workspace.element_size(), _stream(stream))
    _check("up_compact", st)
    return x_out, pos_out, cu_seqlens_out, total_kept, src_idx


def compact_noalloc(x, pos, cu_seqlens, G, keep, cu_blocks, x_out, pos_out, cu_seqlens_out,
                    src_idx, total_kept, stream=None):
    """up_compact without a workspace, for callers that cannot allocate device
    memory: every output buffer must be passed in, and the library's fixed
    scratch is used instead (see up_compact_noalloc in include/up.h).  src_idx
    may be None.  Every tensor's type, dtype and size is checked before its
    device, so a wrong argument raises before anything reaches the library."""
    args = [(x, "x", torch.bfloat16), (pos, "pos", torch.int32),
            (cu_seqlens, "cu_seqlens", torch.int32), (keep, "keep", torch.uint8),
            (cu_blocks, "cu_blocks", torch.int32), (x_out, "x_out", torch.bfloat16),
            (pos_out, "pos_out", torch.int32), (cu_seqlens_out, "cu_seqlens_out", torch.int32),
            (total_kept, "total_kept", torch.int32)]
    if src_idx is not None:
        args.append((src_idx, "src_idx", torch.int32))
    for t, name, dtype in args:
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if x.dim() != 2 or x_out.dim() != 2 or x_out.shape[1] != x.shape[1]:
        raise ValueError("x and x_out must be [rows, hidden] with the same hidden size")
    total, hidden = x.shape
    B = cu_seqlens.numel() - 1
    nb_cap = total // G + B if G > 0 else 0
    if B < 0 or cu_blocks.numel() != B + 1 or cu_seqlens_out.numel() < B + 1:
        raise ValueError("cu_seqlens, cu_blocks and cu_seqlens_out must hold num_seqs + 1 entries")
    if pos.numel() < total or x_out.shape[0] < total or pos_out.numel() < total:
        raise ValueError("pos, x_out and pos_out must hold total_tokens rows")
    if src_idx is not None and src_idx.numel() < total:
        raise ValueError("src_idx must hold total_tokens entries")
    if keep.numel() < min(nb_cap, 1) or total_kept.numel() < 1:
        raise ValueError("keep must hold the block flags and total_kept one entry")
    dev = x.device
    for t, name, dtype in args:
        _need(t, name, dtype, dev)
    st = lib().up_compact_noalloc(_ptr(x), _ptr(pos), hidden, _ptr(cu_seqlens), B, total, G,
                                  _ptr(keep), _ptr(cu_blocks), _ptr(x_out), _ptr(pos_out),
                                  _ptr(cu_seqlens_out), _ptr(src_idx), _ptr(total_kept),
                                  _stream(stream))
    _check("up_compact_noalloc", st)
    return x_out, pos_out, cu_seqlens_out, total_kept, src_idx


def set_kernel_timing_events(start=None, stop=None):
    """Record two torch.cuda.Event objects around the tensor-core scoring kernel
    of every later score_blocks call on this thread (None, None to stop)."""
    h = lambda e: None if e is None else ctypes.c_void_p(e.cuda_event)
    _check("up_set_kernel_timing_events", lib().up_set_kernel_timing_events(h(start), h(stop)))


def measure_ex2_rate(stream=None) -> float:
    """The GPU's sustained MUFU ex2 rate in exponentials per second (a short
    microbenchmark on the current device; synchronises the stream)."""
    v = ctypes.c_double(0.0)
    _check("up_measure_ex2_rate", lib().up_measure_ex2_rate(ctypes.byref(v), _stream(stream)))
    return float(v.value)


def set_wait_limit(cycles: int = 0):
    """Bound, in SM clock cycles, of every spin-wait inside the scoring kernel
    for scoring calls issued after this one (0: the default, about two
    seconds).  For tests of the failure path: an expired wait stops the
    kernel cleanly and sets the timeout bit that get_device_error() reports."""
    _check("up_set_wait_limit", lib().up_set_wait_limit(int(cycles)))


def get_device_error() -> int:
    """Read and clear the library's sticky device error bits (synchronises the device)."""
    v = ctypes.c_uint32(0)
    st = lib().up_get_device_error(ctypes.byref(v))
    if st not in (0, 5, 6):  # OK, or a device bit was set
        raise UpError("up_get_device_error", st)
    return int(v.value)


class Sparsifier:
    """Preallocated buffers for repeated score -> select -> compact passes over
    batches of one shape (the three C-ABI calls, in order, on one stream)."""

    def __init__(self, num_seqs, total_tokens, Hq, Hk, d, hidden, n, G, p, device="cuda"):
        dev = torch.device(device)
        self.num_seqs, self.total, self.n, self.G, self.p = num_seqs, total_tokens, n, G, p
        cap = total_tokens // G + num_seqs
        self.scores = torch.empty(max(cap, 1), dtype=torch.float32, device=dev)
        self.cu_blocks = torch.empty(num_seqs + 1, dtype=torch.int32, device=dev)
        self.keep = torch.empty(max(cap, 1), dtype=torch.uint8, device=dev)
        self.kept_tokens = torch.empty(max(num_seqs, 1), dtype=torch.int32, device=dev)
        self.x_out = torch.empty(max(total_tokens, 1), hidden, dtype=torch.bfloat16, device=dev)
        self.pos_out = torch.empty(max(total_tokens, 1), dtype=torch.int32, device=dev)
        self.cu_out = torch.empty(num_seqs + 1, dtype=torch.int32, device=dev)
        self.src_idx = torch.empty(max(total_tokens, 1), dtype=torch.int32, device=dev)
        self.total_kept = torch.empty(1, dtype=torch.int32, device=dev)
        self.ws_score = _alloc_ws(score_blocks_workspace(num_seqs, total_tokens, Hq, Hk, d, n, G), dev)
        self.ws_compact = _alloc_ws(compact_workspace(num_seqs, total_tokens, G), dev)

    def launches_per_step(self) -> int:
        # score: plan, tensor-core kernel (scores included); select: 1;
        # compact: 1, or index + gather past 16384 possible blocks
        score = 2 if self.total > 0 and self.num_seqs > 0 else 1
        compact = 1 if self.total // self.G + self.num_seqs <= 16384 else 2
        return score + 1 + compact

    def run(self, q_last, k, cu_seqlens, x, pos, stream=None):
        score_blocks(q_last, k, cu_seqlens, self.n, self.G, self.scores, self.cu_blocks,
                     self.ws_score, stream)
        select_topp(self.scores, self.cu_blocks, cu_seqlens, self.G, self.p, self.keep,
                    self.kept_tokens, stream)
        compact(x, pos, cu_seqlens, self.G, self.keep, self.cu_blocks, self.x_out, self.pos_out,
                self.cu_out, self.src_idx, self.total_kept, self.ws_compact, stream)
        return self.total_kept
