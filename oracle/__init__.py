"""fp64 CPU oracle for UniPrefill block scoring, top-p selection and compaction.

TEST INFRASTRUCTURE ONLY: imported by tests/, by the package entry's smoke()
check and by bench.py's CPU-baseline leg, never by the product path.  The
arithmetic lives in ``up_oracle.c`` (plain C, fp64), which shares no code with
the CUDA library.  This module only compiles it with gcc and marshals numpy
arrays through ctypes.

Page citations for every step are in ``up_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "up_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile up_oracle.c into oracle/_build/liboracle.so (plain gcc, no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.orc_token_mass.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, i32]
            lib.orc_token_mass.restype = i32
            lib.orc_block_scores.argtypes = [P, P, i32, i32, P, P]
            lib.orc_block_scores.restype = i32
            lib.orc_select_topp.argtypes = [P, P, P, i32, i32, dbl, P, P, P, P]
            lib.orc_select_topp.restype = i32
            lib.orc_select_topk.argtypes = [P, P, P, i32, i32, i32, P, P]
            lib.orc_select_topk.restype = i32
            lib.orc_keep_last_block.argtypes = [P, P, i32, i32, P, P]
            lib.orc_keep_last_block.restype = i32
            lib.orc_compact.argtypes = [P, P, i64, P, i32, i32, P, P, P, P, P, P]
            lib.orc_compact.restype = i64
            lib.orc_block_csr.argtypes = [P, P, i32, P, P]
            lib.orc_block_csr.restype = i64
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def token_mass(q_last, k, cu_seqlens, Hq, Hk, d, n, nthreads=None):
    """Per-token softmax mass T (fp64, [total_tokens]) of the last n queries.

    q_last: uint16 bf16 bits [sum n_s, Hq, d]; k: uint16 bf16 bits [total, Hk, d].
    """
    lib = _load()
    q_last = _c(q_last, np.uint16)
    k = _c(k, np.uint16)
    cu = _c(cu_seqlens, np.int32)
    B = cu.shape[0] - 1
    mass = np.zeros(int(cu[-1]), dtype=np.float64)
    if nthreads is None:
        nthreads = len(os.sched_getaffinity(0))
    rc = lib.orc_token_mass(_ptr(q_last), _ptr(k), _ptr(cu), B, Hq, Hk, d, n, _ptr(mass),
                            int(nthreads))
    if rc != 0:
        raise ValueError("orc_token_mass rejected its arguments")
    return mass


def block_scores(mass, cu_seqlens, G):
    """Block scores (fp64, [sum nb_s]) and cu_blocks (int32, [B+1]) from token mass."""
    lib = _load()
    mass = _c(mass, np.float64)
    cu = _c(cu_seqlens, np.int32)
    B = cu.shape[0] - 1
    lens = np.diff(cu.astype(np.int64))
    nb_total = int(((lens + G - 1) // G).sum())
    scores = np.zeros(nb_total, dtype=np.float64)
    cu_blocks = np.zeros(B + 1, dtype=np.int32)
    if lib.orc_block_scores(_ptr(mass), _ptr(cu), B, G, _ptr(scores), _ptr(cu_blocks)) != 0:
        raise ValueError("orc_block_scores rejected its arguments")
    return scores, cu_blocks


def score_blocks(q_last, k, cu_seqlens, Hq, Hk, d, n, G, nthreads=None):
    """Token mass followed by block binning: (scores fp64, cu_blocks int32)."""
    return block_scores(token_mass(q_last, k, cu_seqlens, Hq, Hk, d, n, nthreads), cu_seqlens, G)


def select_topp(scores, cu_blocks, cu_seqlens, G, p):
    """Top-p selection.  Returns (keep uint8, kept_tokens int32, cum_incl, cum_excl)."""
    lib = _load()
    scores = _c(scores, np.float64)
    cb = _c(cu_blocks, np.int32)
    cu = _c(cu_seqlens, np.int32)
    B = cu.shape[0] - 1
    nb = scores.shape[0]
    keep = np.zeros(nb, dtype=np.uint8)
    kept = np.zeros(B, dtype=np.int32)
    ci = np.zeros(nb, dtype=np.float64)
    ce = np.zeros(nb, dtype=np.float64)
    rc = lib.orc_select_topp(_ptr(scores), _ptr(cb), _ptr(cu), B, G, float(p), _ptr(keep),
                             _ptr(kept), _ptr(ci), _ptr(ce))
    if rc != 0:
        raise ValueError("orc_select_topp rejected its arguments")
    return keep, kept, ci, ce


def select_topk(scores, cu_blocks, cu_seqlens, G, k):
    """Top-k selection.  Returns (keep uint8, kept_tokens int32)."""
    lib = _load()
    scores = _c(scores, np.float64)
    cb = _c(cu_blocks, np.int32)
    cu = _c(cu_seqlens, np.int32)
    B = cu.shape[0] - 1
    keep = np.zeros(scores.shape[0], dtype=np.uint8)
    kept = np.zeros(B, dtype=np.int32)
    rc = lib.orc_select_topk(_ptr(scores), _ptr(cb), _ptr(cu), B, G, int(k), _ptr(keep), _ptr(kept))
    if rc != 0:
        raise ValueError("orc_select_topk rejected its arguments")
    return keep, kept


def keep_last_block(keep, kept_tokens, cu_blocks, cu_seqlens, G):
    """The keep-last option applied to a selection.  Returns new (keep, kept_tokens)."""
    lib = _load()
    keep = np.array(keep, dtype=np.uint8, copy=True)
    kept = np.array(kept_tokens, dtype=np.int32, copy=True)
    cb = _c(cu_blocks, np.int32)
    cu = _c(cu_seqlens, np.int32)
    rc = lib.orc_keep_last_block(_ptr(cb), _ptr(cu), cu.shape[0] - 1, G, _ptr(keep), _ptr(kept))
    if rc != 0:
        raise ValueError("orc_keep_last_block rejected its arguments")
    return keep, kept


def compact(x, pos, cu_seqlens, G, keep, cu_blocks, with_x=True):
    """Compaction.  Returns (x_out uint16 or None, pos_out, cu_out, src_idx)."""
    lib = _load()
    cu = _c(cu_seqlens, np.int32)
    B = cu.shape[0] - 1
    keep = _c(keep, np.uint8)
    cb = _c(cu_blocks, np.int32)
    pos = _c(pos, np.int32)
    lens = np.diff(cu.astype(np.int64))
    total_kept = 0
    for s in range(B):
        for b in range(int(cb[s + 1] - cb[s])):
            if keep[cb[s] + b]:
                total_kept += int(min(G, lens[s] - b * G))
    hidden = 0
    x_out = None
    if with_x:
        x = _c(x, np.uint16)
        hidden = x.shape[1]
        x_out = np.zeros((total_kept, hidden), dtype=np.uint16)
    pos_out = np.zeros(total_kept, dtype=np.int32)
    cu_out = np.zeros(B + 1, dtype=np.int32)
    src = np.zeros(total_kept, dtype=np.int32)
    got = lib.orc_compact(_ptr(x) if with_x else None, _ptr(pos), hidden, _ptr(cu), B, G,
                          _ptr(keep), _ptr(cb), _ptr(x_out), _ptr(pos_out), _ptr(cu_out),
                          _ptr(src))
    if got != total_kept:
        raise ValueError("orc_compact rejected its arguments")
    return x_out, pos_out, cu_out, src


def block_csr(keep, cu_blocks):
    """Block CSR of the kept blocks.  Returns (indptr int32 [B+1], indices int32 [nnz])."""
    lib = _load()
    keep = _c(keep, np.uint8)
    cb = _c(cu_blocks, np.int32)
    B = cb.shape[0] - 1
    indptr = np.zeros(B + 1, dtype=np.int32)
    indices = np.zeros(max(int(cb[-1]), 1), dtype=np.int32)
    nnz = lib.orc_block_csr(_ptr(keep), _ptr(cb), B, _ptr(indptr), _ptr(indices))
    if nnz < 0:
        raise ValueError("orc_block_csr rejected its arguments")
    return indptr, indices[:nnz]
