"""Pins for the fp64 oracle against facts fixed by the pages and by mathematics.

Nothing here compares the oracle with itself or with the CUDA path.  Each pin is
a closed form, an invariant, a hand-enumerated case, a brute force over tiny
inputs, or a special case that reduces to a library routine (fp64 torch/scipy
softmax), chosen so that a dropped term, a wrong sign or index, a transposed
operand, a wrong scale or a wrong causal convention fails at least one.
"""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from block_sparse_long_up_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(a):
    return synth.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def _f64(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def _random_case(lens, Hq, Hk, d, n, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    cu = np.zeros(len(lens) + 1, np.int32)
    cu[1:] = np.cumsum(lens)
    nq = sum(min(n, L) for L in lens)
    q = _bits(rng.standard_normal((nq, Hq, d)) * scale)
    k = _bits(rng.standard_normal((int(cu[-1]), Hk, d)) * scale)
    return q, k, cu


# --------------------------------------------------------------------------
# token mass / block scores
# --------------------------------------------------------------------------

def test_two_key_hand_worked():
    """One query at position 1, two keys, d=4: z = (0, 4/sqrt(4)) = (0, 2).

    Softmax by hand: P = (1/(1+e^2), e^2/(1+e^2)).  With scale 1/d instead of
    1/sqrt(d) this would be (1/(1+e), e/(1+e)); with a strict causal mask the
    query would see key 0 only.
    """
    q = _bits([[[1, 1, 1, 1]]])               # [n=1, Hq=1, d=4]
    k = _bits([[[0, 0, 0, 0]], [[1, 1, 1, 1]]])  # [L=2, Hk=1, d=4]
    cu = np.array([0, 2], np.int32)
    mass = oracle.token_mass(q, k, cu, 1, 1, 4, 1, nthreads=1)
    e2 = math.exp(2.0)
    assert mass[0] == pytest.approx(1.0 / (1.0 + e2), rel=1e-14)
    assert mass[1] == pytest.approx(e2 / (1.0 + e2), rel=1e-14)
    sc, cb = oracle.block_scores(mass, cu, 2)
    assert cb.tolist() == [0, 1] and sc[0] == pytest.approx(1.0, rel=1e-15)


def test_two_queries_hand_worked():
    """n=2 on L=2: query 0 (position 0) sees key 0 only, so P = (1, 0); query 1 as above.

    The mass is averaged over the n_s = 2 queries: T = ((1 + 1/(1+e^2))/2, (e^2/(1+e^2))/2).
    """
    q = _bits([[[5, -3, 2, 7]], [[1, 1, 1, 1]]])
    k = _bits([[[0, 0, 0, 0]], [[1, 1, 1, 1]]])
    cu = np.array([0, 2], np.int32)
    mass = oracle.token_mass(q, k, cu, 1, 1, 4, 2, nthreads=1)
    e2 = math.exp(2.0)
    assert mass[0] == pytest.approx((1.0 + 1.0 / (1.0 + e2)) / 2.0, rel=1e-14)
    assert mass[1] == pytest.approx((e2 / (1.0 + e2)) / 2.0, rel=1e-14)


@pytest.mark.parametrize("lens,n", [([37], 8), ([5, 64, 3], 16), ([100, 7], 100), ([2, 1], 4)])
def test_closed_form_zero_queries(lens, n):
    """q == 0 makes every visible logit 0, so query t spreads 1/(a_t+1) over keys 0..a_t.

    T_i = (1/n_s) * sum_{t : a_t >= i} 1/(a_t + 1), identical for every head.
    """
    Hq, Hk, d = 4, 2, 8
    _, k, cu = _random_case(lens, Hq, Hk, d, n, seed=3)
    nq = sum(min(n, L) for L in lens)
    q = np.zeros((nq, Hq, d), np.uint16)
    mass = oracle.token_mass(q, k, cu, Hq, Hk, d, n, nthreads=2)
    for s, L in enumerate(lens):
        ns = min(n, L)
        want = np.zeros(L)
        for t in range(ns):
            a = L - ns + t
            want[: a + 1] += 1.0 / (a + 1)
        want /= ns
        np.testing.assert_allclose(mass[cu[s]:cu[s + 1]], want, rtol=1e-12, atol=0)


@pytest.mark.parametrize("lens,Hq,Hk,d,n,G", [
    ([64], 2, 1, 16, 8, 16),
    ([50, 33], 4, 2, 8, 12, 16),     # ragged last blocks
    ([9, 120, 1], 6, 3, 32, 20, 32),
    ([17], 3, 3, 12, 17, 5),         # n == L, G does not divide L
])
def test_dense_torch_softmax(lens, Hq, Hk, d, n, G):
    """Tiny shapes against fp64 torch.softmax of the masked logit matrix.

    Logits are Q K^T / sqrt(d) built from the same bf16 values; keys after each
    query's absolute position are masked (-inf) as in a causal prefill.
    """
    q, k, cu = _random_case(lens, Hq, Hk, d, n, seed=11, scale=2.0)
    sc, cb = oracle.score_blocks(q, k, cu, Hq, Hk, d, n, G, nthreads=3)
    qf = torch.from_numpy(_f64(q))
    kf = torch.from_numpy(_f64(k))
    qoff = 0
    g = Hq // Hk
    for s, L in enumerate(lens):
        ns = min(n, L)
        qs = qf[qoff:qoff + ns]              # [ns, Hq, d]
        ks = kf[cu[s]:cu[s + 1]]             # [L, Hk, d]
        kr = ks.repeat_interleave(g, dim=1)  # [L, Hq, d]
        logits = torch.einsum("thc,ihc->hti", qs, kr) / math.sqrt(d)
        apos = torch.arange(L - ns, L).view(1, ns, 1)
        keys = torch.arange(L).view(1, 1, L)
        logits = logits.masked_fill(keys > apos, float("-inf"))
        P = torch.softmax(logits, dim=-1)    # [Hq, ns, L]
        T = P.sum(dim=(0, 1)) / (ns * Hq)
        nb = (L + G - 1) // G
        padded = torch.zeros(nb * G, dtype=torch.float64)
        padded[:L] = T
        want = padded.view(nb, G).sum(dim=1).numpy()
        np.testing.assert_allclose(sc[cb[s]:cb[s + 1]], want, rtol=1e-12, atol=1e-15)
        qoff += ns


def test_single_row_scipy_softmax():
    """n=1, Hq=1: the mass is one softmax row, computed here with scipy."""
    L, d = 300, 24
    q, k, cu = _random_case([L], 1, 1, d, 1, seed=5, scale=3.0)
    mass = oracle.token_mass(q, k, cu, 1, 1, d, 1, nthreads=1)
    z = _f64(k)[:, 0, :] @ _f64(q)[0, 0, :] / math.sqrt(d)
    np.testing.assert_allclose(mass, scipy.special.softmax(z), rtol=1e-12, atol=1e-300)


@pytest.mark.parametrize("lens", [[200], [64, 129, 1, 70]])
def test_scores_sum_to_one(lens):
    q, k, cu = _random_case(lens, 4, 1, 16, 32, seed=9, scale=2.5)
    sc, cb = oracle.score_blocks(q, k, cu, 4, 1, 16, 32, 16)
    for s in range(len(lens)):
        assert abs(sc[cb[s]:cb[s + 1]].sum() - 1.0) <= 1e-12


def test_g1_is_token_mass_and_large_g_is_one_block():
    lens = [77, 40]
    q, k, cu = _random_case(lens, 2, 2, 8, 10, seed=21)
    mass = oracle.token_mass(q, k, cu, 2, 2, 8, 10)
    sc1, cb1 = oracle.block_scores(mass, cu, 1)
    np.testing.assert_array_equal(sc1, mass)
    assert cb1.tolist() == [0, 77, 117]
    scL, cbL = oracle.block_scores(mass, cu, 128)
    assert cbL.tolist() == [0, 1, 2]
    np.testing.assert_allclose(scL, [1.0, 1.0], rtol=0, atol=1e-12)


def test_gqa_equals_mha_with_repeated_kv_heads():
    """Query head h reads KV head h // (Hq/Hk): GQA equals MHA over contiguously repeated KV heads."""
    lens, Hq, Hk, d, n = [90, 33], 6, 2, 16, 12
    q, k, cu = _random_case(lens, Hq, Hk, d, n, seed=13, scale=2.0)
    gqa = oracle.token_mass(q, k, cu, Hq, Hk, d, n)
    k_rep = np.repeat(k, Hq // Hk, axis=1)
    mha = oracle.token_mass(q, k_rep, cu, Hq, Hq, d, n)
    np.testing.assert_array_equal(gqa, mha)
    # the other plausible mapping (h % Hk) gives a different answer on these inputs
    k_tile = np.tile(k, (1, Hq // Hk, 1))
    wrong = oracle.token_mass(q, k_tile, cu, Hq, Hq, d, n)
    assert np.max(np.abs(wrong - gqa)) > 1e-6


def test_dominant_key_takes_its_block():
    L, d, G, n = 256, 32, 16, 8
    rng = np.random.default_rng(1)
    qv = rng.standard_normal((n, 1, d))
    kv = rng.standard_normal((L, 1, d)) * 0.1
    kv[37, 0, :] = 4.0 * qv.mean(axis=0)[0] / np.linalg.norm(qv.mean(axis=0)[0]) * math.sqrt(d)
    qv = qv / np.linalg.norm(qv, axis=-1, keepdims=True) * math.sqrt(d) * 3
    q, k = _bits(qv), _bits(kv)
    cu = np.array([0, L], np.int32)
    sc, _ = oracle.score_blocks(q, k, cu, 1, 1, d, n, G)
    assert np.argmax(sc) == 37 // G and sc[37 // G] > 0.99


# --------------------------------------------------------------------------
# top-p selection
# --------------------------------------------------------------------------

def _load_topp_golden():
    cases = []
    with open(os.path.join(GOLDEN, "topp_hand_enumerated.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            p, scores, kept = (part.strip() for part in line.split(";"))
            cases.append((float(p), [float(v) for v in scores.split(",")],
                          sorted(int(v) for v in kept.split(","))))
    return cases


@pytest.mark.parametrize("p,scores,kept", _load_topp_golden())
def test_topp_hand_enumerated(p, scores, kept):
    nb = len(scores)
    G = 4
    cu = np.array([0, nb * G], np.int32)
    cb = np.array([0, nb], np.int32)
    keep, kt, _, _ = oracle.select_topp(np.array(scores), cb, cu, G, p)
    assert sorted(np.nonzero(keep)[0].tolist()) == kept
    assert kt.tolist() == [len(kept) * G]


@pytest.mark.parametrize("seed", range(6))
def test_topp_brute_force(seed):
    """For nb <= 12: the kept set has the fewest blocks of any subset with mass >= p,
    and the largest mass among subsets of that size."""
    rng = np.random.default_rng(100 + seed)
    nb = int(rng.integers(1, 13))
    raw = rng.exponential(size=nb) ** 3
    scores = raw / raw.sum()
    p = float(rng.uniform(0.05, 0.999))
    G = 8
    L = nb * G - int(rng.integers(0, G))  # ragged last block
    cu = np.array([0, L], np.int32)
    cb = np.array([0, nb], np.int32)
    keep, kt, _, _ = oracle.select_topp(scores, cb, cu, G, p)
    kept = set(np.nonzero(keep)[0].tolist())
    best_k = None
    for r in range(1, nb + 1):
        if any(scores[list(c)].sum() >= p for c in itertools.combinations(range(nb), r)):
            best_k = r
            break
    if best_k is None:  # rounding left the total short of p: everything is kept
        assert kept == set(range(nb))
        return
    assert len(kept) == best_k
    best_mass = max(scores[list(c)].sum() for c in itertools.combinations(range(nb), best_k))
    assert scores[sorted(kept)].sum() == pytest.approx(best_mass, rel=1e-12)
    lens = [min(G, L - b * G) for b in range(nb)]
    assert kt[0] == sum(lens[b] for b in kept)


def test_topp_p_one_keeps_everything_and_tiny_p_keeps_the_top_block():
    rng = np.random.default_rng(7)
    scores = rng.random(50)
    scores /= scores.sum()
    cb = np.array([0, 50], np.int32)
    cu = np.array([0, 50 * 4 - 3], np.int32)
    keep, kt, _, _ = oracle.select_topp(scores, cb, cu, 4, 1.0)
    assert keep.all() and kt[0] == 197
    keep, _, _, _ = oracle.select_topp(scores, cb, cu, 4, 1e-12)
    assert np.nonzero(keep)[0].tolist() == [int(np.argmax(scores))]


def test_topp_zero_queries_keeps_lowest_indices():
    """With q == 0 every block that ends before the query window has the same
    score (bitwise) and the window's blocks score lower, so top-p keeps a prefix
    of block indices: the tie rule at scale."""
    L, n, G, Hq, Hk, d = 1024, 64, 16, 2, 1, 8
    _, k, cu = _random_case([L], Hq, Hk, d, n, seed=2)
    q = np.zeros((n, Hq, d), np.uint16)
    sc, cb = oracle.score_blocks(q, k, cu, Hq, Hk, d, n, G)
    first_window_block = (L - n) // G
    assert len(set(sc[:first_window_block].tolist())) == 1
    assert np.all(sc[first_window_block:] < sc[0])
    for p in (0.3, 0.5, 0.9):
        keep, _, _, _ = oracle.select_topp(sc, cb, cu, G, p)
        idx = np.nonzero(keep)[0]
        assert idx.tolist() == list(range(len(idx)))


def test_topp_cumulative_band_outputs():
    scores = np.array([0.5, 0.25, 0.125, 0.125])
    keep, _, ci, ce = oracle.select_topp(scores, np.array([0, 4], np.int32),
                                         np.array([0, 16], np.int32), 4, 0.8)
    np.testing.assert_array_equal(ci, [0.5, 0.75, 0.875, 1.0])
    np.testing.assert_array_equal(ce, [0.0, 0.5, 0.75, 0.875])


# --------------------------------------------------------------------------
# top-k selection and the keep-last option
# --------------------------------------------------------------------------

def _load_topk_golden():
    cases = []
    with open(os.path.join(GOLDEN, "topk_hand_enumerated.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, scores, kept = (part.strip() for part in line.split(";"))
            cases.append((int(k), [float(v) for v in scores.split(",")],
                          sorted(int(v) for v in kept.split(","))))
    return cases


@pytest.mark.parametrize("k,scores,kept", _load_topk_golden())
def test_topk_hand_enumerated(k, scores, kept):
    nb, G = len(scores), 4
    keep, kt = oracle.select_topk(np.array(scores), np.array([0, nb], np.int32),
                                  np.array([0, nb * G], np.int32), G, k)
    assert sorted(np.nonzero(keep)[0].tolist()) == kept
    assert kt.tolist() == [len(kept) * G]


@pytest.mark.parametrize("seed", range(8))
def test_topk_brute_force(seed):
    """For nb <= 12, with scores drawn from a few values (many ties): the kept set
    is the lexicographically smallest (sorted indices) among the k-subsets of
    largest total score, which is what ranking with ties to the lower index picks."""
    rng = np.random.default_rng(300 + seed)
    nb = int(rng.integers(1, 13))
    scores = rng.choice(np.array([0.5, 0.25, 0.125, 0.0625]), size=nb)
    k = int(rng.integers(1, nb + 3))
    G = 8
    L = nb * G - int(rng.integers(0, G))
    keep, kt = oracle.select_topk(scores, np.array([0, nb], np.int32),
                                  np.array([0, L], np.int32), G, k)
    m = min(k, nb)
    best = max(scores[list(c)].sum() for c in itertools.combinations(range(nb), m))
    cands = [c for c in itertools.combinations(range(nb), m) if scores[list(c)].sum() == best]
    assert tuple(np.nonzero(keep)[0].tolist()) == min(cands)
    lens = [min(G, L - b * G) for b in range(nb)]
    assert kt[0] == sum(lens[b] for b in np.nonzero(keep)[0])


def test_topk_zero_queries_keeps_lowest_indices():
    """q == 0: equal scores before the query window, lower inside it; top-k keeps
    the first k block indices (the tie rule at scale)."""
    L, n, G, Hq, Hk, d = 1024, 64, 16, 2, 1, 8
    _, k, cu = _random_case([L], Hq, Hk, d, n, seed=2)
    q = np.zeros((n, Hq, d), np.uint16)
    sc, cb = oracle.score_blocks(q, k, cu, Hq, Hk, d, n, G)
    for kk in (1, 7, 30):
        keep, _ = oracle.select_topk(sc, cb, cu, G, kk)
        assert np.nonzero(keep)[0].tolist() == list(range(kk))


def test_keep_last_block_option():
    """The keep-last step keeps each non-empty sequence's last block (ragged length
    counted) and leaves a selection that already holds it unchanged."""
    lens = [37, 64, 0, 5]
    G = 16
    cu = np.array([0] + list(np.cumsum(lens)), np.int32)
    nbs = [(L + G - 1) // G for L in lens]
    cb = np.array([0] + list(np.cumsum(nbs)), np.int32)
    keep = np.zeros(int(cb[-1]), np.uint8)
    keep[0] = 1                    # sequence 0: first block only
    keep[int(cb[1]) + 3] = 1       # sequence 1: already holds its last block
    kept = np.array([16, 16, 0, 0], np.int32)
    k2, t2 = oracle.keep_last_block(keep, kept, cb, cu, G)
    assert k2[int(cb[1]) - 1] == 1 and t2[0] == 16 + (37 - 2 * 16)
    assert t2[1] == 16 and k2[int(cb[1]):int(cb[2])].tolist() == [0, 0, 0, 1]
    assert t2[2] == 0
    assert k2[int(cb[3])] == 1 and t2[3] == 5


# --------------------------------------------------------------------------
# compaction
# --------------------------------------------------------------------------

def _compact_case(lens, G, hidden, seed, keep_prob):
    rng = np.random.default_rng(seed)
    cu = np.zeros(len(lens) + 1, np.int32)
    cu[1:] = np.cumsum(lens)
    nbs = [(L + G - 1) // G for L in lens]
    cb = np.zeros(len(lens) + 1, np.int32)
    cb[1:] = np.cumsum(nbs)
    keep = (rng.random(int(cb[-1])) < keep_prob).astype(np.uint8)
    x = rng.integers(0, 1 << 16, size=(int(cu[-1]), hidden), dtype=np.uint16)
    pos = np.concatenate([np.arange(L, dtype=np.int32) for L in lens])
    return cu, cb, keep, x, pos


def test_compact_keep_all_is_identity():
    lens, G = [70, 3, 128], 16
    cu, cb, keep, x, pos = _compact_case(lens, G, 24, 0, 1.1)
    assert keep.all()
    x_out, pos_out, cu_out, src = oracle.compact(x, pos, cu, G, keep, cb)
    np.testing.assert_array_equal(x_out, x)
    np.testing.assert_array_equal(pos_out, pos)
    np.testing.assert_array_equal(cu_out, cu)
    np.testing.assert_array_equal(src, np.arange(cu[-1]))


@pytest.mark.parametrize("seed", range(3))
def test_compact_invariants(seed):
    lens, G = [70, 0, 3, 128, 65], 16
    cu, cb, keep, x, pos = _compact_case(lens, G, 40, seed, 0.4)
    x_out, pos_out, cu_out, src = oracle.compact(x, pos, cu, G, keep, cb)
    # each output row is a copy of its source row, position included
    np.testing.assert_array_equal(x_out, x[src])
    np.testing.assert_array_equal(pos_out, pos[src])
    # source rows strictly increase: original order is kept
    assert np.all(np.diff(src) > 0)
    # exactly the rows of kept blocks appear: a per-token mask, each token
    # looking up its own block's flag (token-centric, where the oracle walks
    # the blocks)
    tok = np.arange(int(cu[-1]))
    seq = np.searchsorted(cu, tok, side="right") - 1
    mask = keep[cb[seq] + (tok - cu[seq]) // G].astype(bool)
    np.testing.assert_array_equal(src, np.nonzero(mask)[0])
    np.testing.assert_array_equal(np.diff(cu_out), np.bincount(seq[mask], minlength=len(lens)))
    # cu_out is monotone, and positions strictly increase within each output sequence
    assert np.all(np.diff(cu_out) >= 0) and cu_out[-1] == len(src)
    for s in range(len(lens)):
        assert np.all(np.diff(pos_out[cu_out[s]:cu_out[s + 1]]) > 0)


def test_compact_hand_example():
    """Two sequences of 5 and 3 tokens, G = 2: blocks {0,1} {2,3} {4} and
    {5,6} {7}; keeping blocks 0 and 2 of the first and block 1 of the second
    keeps tokens 0, 1, 4 and 7, positions gathered unchanged."""
    cu = np.array([0, 5, 8], np.int32)
    cb = np.array([0, 3, 5], np.int32)
    keep = np.array([1, 0, 1, 0, 1], np.uint8)
    x = np.arange(8 * 8, dtype=np.uint16).reshape(8, 8)
    pos = np.array([10, 11, 12, 13, 14, 0, 1, 2], np.int32)
    x_out, pos_out, cu_out, src = oracle.compact(x, pos, cu, 2, keep, cb)
    assert src.tolist() == [0, 1, 4, 7]
    assert pos_out.tolist() == [10, 11, 14, 2]
    assert cu_out.tolist() == [0, 3, 4]
    np.testing.assert_array_equal(x_out, x[[0, 1, 4, 7]])


def test_block_csr_hand_example_and_round_trip():
    """Block CSR (FlashPrefill V2 review, key-terms section): a hand-written
    case with an empty sequence and a sequence that keeps nothing, then random
    batches whose CSR must rebuild the keep flags exactly."""
    keep = np.array([1, 0, 1, 0, 0, 1, 1, 1, 0], np.uint8)
    cb = np.array([0, 3, 3, 5, 9], np.int32)
    indptr, indices = oracle.block_csr(keep, cb)
    assert indptr.tolist() == [0, 2, 2, 2, 5]
    assert indices.tolist() == [0, 2, 0, 1, 2]
    rng = np.random.default_rng(0)
    for _ in range(20):
        nbs = rng.integers(0, 40, size=rng.integers(1, 8))
        cb = np.concatenate([[0], np.cumsum(nbs)]).astype(np.int32)
        keep = (rng.random(int(cb[-1])) < rng.random()).astype(np.uint8)
        indptr, indices = oracle.block_csr(keep, cb)
        assert indptr[-1] == keep.sum() and np.all(np.diff(indptr) >= 0)
        rebuilt = np.zeros_like(keep)
        for s in range(len(nbs)):
            row = indices[indptr[s]:indptr[s + 1]]
            assert np.all(np.diff(row) > 0) and np.all((row >= 0) & (row < nbs[s]))
            rebuilt[cb[s] + row] = 1
        assert np.array_equal(rebuilt, keep)
