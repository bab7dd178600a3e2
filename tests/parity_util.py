"""Helpers shared by the GPU parity tests: moving synthetic inputs to the device,
running the three C-ABI calls, and the comparison contract.

Comparison contract (numbers fixed by the benchmark spec of this library):
  * block scores: |gpu - oracle| <= max(1e-3 * |oracle|, 1e-6) for every block;
  * kept sets: bit-exact, except blocks whose oracle cumulative mass at their
    rank (inclusive or exclusive) lies within 1e-4 of p -- those are counted,
    not failed;
  * compaction on the same keep flags: bit-exact x_out, pos_out, cu_seqlens_out
    and src_idx.
"""
from __future__ import annotations

import logging
import os

import numpy as np
import torch

import block_sparse_long_up_gb300 as up
import oracle

SCORE_RTOL = 1e-3
SCORE_ATOL = 1e-6
BAND = 1e-4

# every full_check's report, in order: tests/conftest.py prints them in the
# terminal summary, so a quiet run still shows the worst score error and the
# excused kept-set count of each case
REPORTS: list = []
log = logging.getLogger("parity")


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def to_dev_i32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def gpu_scores(inp, n, G):
    q = to_dev_bf16(inp.q_last)
    k = to_dev_bf16(inp.k)
    cu = to_dev_i32(inp.cu_seqlens)
    sc, cb = up.score_blocks(q, k, cu, n, G)
    torch.cuda.synchronize()
    cbh = cb.cpu().numpy()
    return sc[: int(cbh[-1])].cpu().numpy().astype(np.float64), cbh


def score_failures(gpu, orc):
    tol = np.maximum(SCORE_RTOL * np.abs(orc), SCORE_ATOL)
    bad = np.abs(gpu - orc) > tol
    return int(bad.sum()), float(np.max(np.abs(gpu - orc) / np.maximum(np.abs(orc), 1e-30)))


def keep_mismatch(gpu_keep, orc_keep, cum_incl, cum_excl, p):
    """(hard failures, excused-in-band count)."""
    diff = gpu_keep.astype(bool) != orc_keep.astype(bool)
    in_band = (np.abs(cum_incl - p) <= BAND) | (np.abs(cum_excl - p) <= BAND)
    return int((diff & ~in_band).sum()), int((diff & in_band).sum())


def gpu_select(scores_np, cb_np, cu_np, G, p):
    sc = torch.from_numpy(np.ascontiguousarray(scores_np, dtype=np.float32)).cuda()
    keep, kt = up.select_topp(sc, to_dev_i32(cb_np), to_dev_i32(cu_np), G, p)
    torch.cuda.synchronize()
    B = len(cu_np) - 1
    return keep[: len(scores_np)].cpu().numpy(), kt[:B].cpu().numpy()


def gpu_compact(x_bits, pos, cu_np, G, keep_np, cb_np):
    x = to_dev_bf16(x_bits)
    xo, po, cuo, tk, src = up.compact(x, to_dev_i32(pos), to_dev_i32(cu_np), G,
                                      torch.from_numpy(np.ascontiguousarray(keep_np, np.uint8)).cuda(),
                                      to_dev_i32(cb_np))
    torch.cuda.synchronize()
    T = int(tk.item())
    return (xo[:T].view(torch.int16).cpu().numpy().view(np.uint16), po[:T].cpu().numpy(),
            cuo.cpu().numpy(), src[:T].cpu().numpy(), T)


def full_check(inp, n, G, p, check_x=True, nthreads=None):
    """Score + select + compact on the GPU against the oracle; returns a report dict
    and asserts the contract."""
    orc_sc, orc_cb = oracle.score_blocks(inp.q_last, inp.k, inp.cu_seqlens, inp.Hq, inp.Hk,
                                         inp.d, n, G, nthreads=nthreads)
    g_sc, g_cb = gpu_scores(inp, n, G)
    np.testing.assert_array_equal(g_cb, orc_cb)
    nbad, worst = score_failures(g_sc, orc_sc)
    assert nbad == 0, f"{nbad} block scores out of tolerance (worst rel {worst:.3g})"
    for s in range(inp.num_seqs):
        seg = g_sc[orc_cb[s]:orc_cb[s + 1]]
        if len(seg):
            assert abs(seg.sum() - 1.0) <= 1e-4
    orc_keep, orc_kt, ci, ce = oracle.select_topp(orc_sc, orc_cb, inp.cu_seqlens, G, p)
    g_keep, g_kt = gpu_select(g_sc, g_cb, inp.cu_seqlens, G, p)
    hard, excused = keep_mismatch(g_keep, orc_keep, ci, ce, p)
    assert hard == 0, f"{hard} kept-set mismatches outside the {BAND} band"
    # the GPU's own selection on its own scores must agree with the oracle's
    # rule applied to the same fp32 scores
    ref_keep, ref_kt, ci2, ce2 = oracle.select_topp(g_sc.astype(np.float32).astype(np.float64),
                                                    g_cb, inp.cu_seqlens, G, p)
    hard2, _ = keep_mismatch(g_keep, ref_keep, ci2, ce2, p)
    assert hard2 == 0
    max_abs = float(np.max(np.abs(g_sc - orc_sc))) if len(g_sc) else 0.0
    report = dict(excused=excused, worst_rel=worst, max_abs=max_abs, kept=int(g_keep.sum()),
                  blocks=len(g_keep), n=n, G=G, p=p)
    if check_x and inp.x is not None:
        xo, po, cuo, src, T = gpu_compact(inp.x, inp.pos, inp.cu_seqlens, G, g_keep, g_cb)
        ox, opos, ocu, osrc = oracle.compact(inp.x, inp.pos, inp.cu_seqlens, G, g_keep, g_cb)
        assert T == len(opos)
        np.testing.assert_array_equal(cuo, ocu)
        np.testing.assert_array_equal(src, osrc)
        np.testing.assert_array_equal(po, opos)
        assert np.array_equal(xo, ox)
        report["kept_tokens"] = T
    report["case"] = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    REPORTS.append(report)
    log.info("parity %s", report)
    return report
