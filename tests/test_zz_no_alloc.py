"""up_compact_noalloc: compaction for callers that cannot allocate device memory.

Such callers (an engine that has already reserved nearly all HBM for its KV
cache, or a serving loop that must not call cudaMalloc because it can
synchronise the device) get this entry point, which uses a fixed scratch array
inside the library instead of a workspace.  These tests call it through the C
ABI twice in a row, with different batches large enough to need the scratch,
and require its outputs to equal those of up_compact (compaction is a bit
copy, so equal means bit-exact).  The second call has fewer kept blocks than
the first, so a result built from the first call's leftover scratch would
show up.

This file is collected last so that a run stopping at its first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import block_sparse_long_up_gb300 as up

pytestmark = pytest.mark.gpu


def _batch(lens, G, hidden, keep_prob, seed):
    rng = np.random.default_rng(seed)
    cu = np.zeros(len(lens) + 1, np.int32)
    cu[1:] = np.cumsum(lens)
    nbs = [(L + G - 1) // G for L in lens]
    cb = np.zeros(len(lens) + 1, np.int32)
    cb[1:] = np.cumsum(nbs)
    keep = (rng.random(int(cb[-1])) < keep_prob).astype(np.uint8)
    x = rng.integers(0, 1 << 16, size=(int(cu[-1]), hidden), dtype=np.uint16)
    pos = rng.integers(0, 1 << 30, size=int(cu[-1])).astype(np.int32)
    dev = torch.device("cuda")
    return dict(
        x=torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev),
        pos=torch.from_numpy(pos).to(dev), cu=torch.from_numpy(cu).to(dev),
        keep=torch.from_numpy(keep).to(dev), cb=torch.from_numpy(cb).to(dev),
        B=len(lens), total=int(cu[-1]), hidden=hidden, G=G)


def _noalloc_via_c_abi(b):
    L = up.lib()
    dev = b["x"].device
    total, hidden = b["total"], b["hidden"]
    x_out = torch.full((max(total, 1), hidden), 7, dtype=torch.bfloat16, device=dev)
    pos_out = torch.full((max(total, 1),), -1, dtype=torch.int32, device=dev)
    cu_out = torch.full((b["B"] + 1,), -1, dtype=torch.int32, device=dev)
    src = torch.full((max(total, 1),), -1, dtype=torch.int32, device=dev)
    tk = torch.full((1,), -1, dtype=torch.int32, device=dev)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = L.up_compact_noalloc(p(b["x"]), p(b["pos"]), hidden, p(b["cu"]), b["B"], total, b["G"],
                              p(b["keep"]), p(b["cb"]), p(x_out), p(pos_out), p(cu_out), p(src),
                              p(tk), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, L.up_status_string(st)
    return x_out, pos_out, cu_out, src, tk


def _same_as_up_compact(b):
    xo, po, cuo, src, tk = _noalloc_via_c_abi(b)
    rx, rp, rcu, rtk, rsrc = up.compact(b["x"], b["pos"], b["cu"], b["G"], b["keep"], b["cb"])
    torch.cuda.synchronize()
    T = int(rtk.item())
    assert int(tk.item()) == T
    assert torch.equal(cuo, rcu)
    assert torch.equal(po[:T], rp[:T])
    assert torch.equal(src[:T], rsrc[:T])
    assert torch.equal(xo[:T].view(torch.int16), rx[:T].view(torch.int16))
    return T


def test_noalloc_matches_up_compact_on_two_calls_in_a_row():
    """Both batches can hold more blocks than the one-kernel compaction takes
    (16384), so both calls go through the library's fixed scratch array."""
    assert torch.cuda.is_available()
    up.build()
    first = _batch([150000, 0, 129, 140000, 77], 16, 64, 0.6, seed=1)   # up to 18142 blocks
    second = _batch([513, 280000, 5], 16, 24, 0.2, seed=2)              # up to 17532 blocks
    t1 = _same_as_up_compact(first)
    t2 = _same_as_up_compact(second)
    assert t1 > t2 > 0
    assert up.get_device_error() == 0


def test_noalloc_small_batch():
    """A batch within the one-kernel limit needs no scratch at all; the entry
    point gives up_compact's result there too."""
    up.build()
    b = _batch([3000, 0, 129, 4096, 77], 64, 4096, 0.6, seed=4)
    assert _same_as_up_compact(b) > 0
    assert up.get_device_error() == 0


def test_noalloc_rejects_batches_beyond_its_scratch():
    up.build()
    L = up.lib()
    b = _batch([64], 64, 16, 1.0, seed=3)
    too_many_tokens = 64 * 65536  # 65536 blocks + 1 sequence: one block over the limit
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = L.up_compact_noalloc(p(b["x"]), p(b["pos"]), 16, p(b["cu"]), 1, too_many_tokens, 64,
                              p(b["keep"]), p(b["cb"]), p(b["x"]), p(b["pos"]), p(b["cu"]), None,
                              p(b["cu"]), None)
    assert st == 3  # UP_ERR_WORKSPACE: nothing launched
