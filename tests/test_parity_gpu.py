"""GPU parity: the C-ABI CUDA path against the fp64 oracle on the same seeded inputs."""
import os

import numpy as np
import pytest
import torch

import block_sparse_long_up_gb300 as up
import oracle
from block_sparse_long_up_gb300 import synth

from parity_util import (full_check, gpu_compact, gpu_scores, gpu_select, keep_mismatch,
                         score_failures, to_dev_bf16, to_dev_i32)

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    up.build()
    up.lib()
    yield
    assert up.get_device_error() == 0


@pytest.mark.parametrize("lens,Hq,Hk,d,n,G,p,gain", [
    ([300], 4, 1, 64, 16, 16, 0.9, 5.0),
    ([1000, 37, 513], 8, 2, 128, 64, 64, 0.95, 5.0),     # ragged tails, several chunks
    ([5, 1, 129], 4, 4, 64, 128, 32, 0.99, 5.0),         # L < n, L == 1
    ([2048], 16, 2, 256, 100, 128, 0.9, 5.0),            # d=256, g=8, 800 rows (ragged tile)
    ([700, 4096], 32, 8, 128, 128, 256, 0.99, 5.0),
    ([777], 2, 1, 128, 1, 64, 0.5, 5.0),                 # one query
    ([3000, 1500], 8, 2, 64, 128, 64, 0.99, None),       # literal unit shift: dense regime
    ([9000], 12, 4, 128, 48, 16, 0.999, 5.0),            # G=16, many blocks per chunk
    ([300, 129, 4100], 4, 1, 64, 16, 256, 0.9, 5.0),     # G=256 block cut short by the sequence end
    ([20000], 8, 1, 256, 96, 128, 0.95, 5.0),            # d=256, 768 rows = 1.5 tile pairs
])
def test_small_shapes(lens, Hq, Hk, d, n, G, p, gain):
    inp = synth.make_inputs(lens, Hq, Hk, d, n, 0.05, gain=gain, hidden=64, seed=sum(lens) + d)
    full_check(inp, n, G, p)


@pytest.mark.parametrize("lens,Hq,Hk,d,n,G,p", [
    ([3000, 700], 16, 1, 128, 1024, 64, 0.95),   # n = 1024 (the largest window), g = 16, L < n
    ([2000], 32, 2, 64, 1024, 32, 0.9),          # g = 16 at head_dim 64: 128 row tiles per head
    ([1500, 1], 48, 3, 256, 1024, 128, 0.99),    # g = 16 at head_dim 256, a one-token sequence
])
def test_largest_window_and_group(lens, Hq, Hk, d, n, G, p):
    """The API's largest query window (n = 1024) and GQA group (Hq / Hk = 16):
    a tile then holds 8 queries of 16 heads, a KV head has up to 128 row tiles,
    and sequences shorter than the window use all of their tokens as queries."""
    inp = synth.make_inputs(lens, Hq, Hk, d, n, 0.05, gain=5.0, hidden=32, seed=sum(lens) + n)
    full_check(inp, n, G, p)


@pytest.mark.parametrize("gain", [5.0, None])
def test_gqa8x2_d64_4k_workload(gain):
    inp = synth.make_workload("gqa8x2_d64_4k", gain=gain)
    w = synth.WORKLOADS["gqa8x2_d64_4k"]
    rep = full_check(inp, w["n"], w["G"], w["p"])
    if gain is not None:
        assert rep["kept"] < rep["blocks"] // 4


def test_scores_are_deterministic():
    inp = synth.make_inputs([5000, 3000], 8, 2, 128, 128, 0.05, seed=3)
    a, _ = gpu_scores(inp, 128, 64)
    b, _ = gpu_scores(inp, 128, 64)
    assert np.array_equal(a, b)


def test_empty_batch_and_empty_sequences():
    inp = synth.make_inputs([0, 300, 0, 65, 0], 4, 2, 64, 32, 0.05, hidden=16, seed=4)
    full_check(inp, 32, 64, 0.9)
    # no sequences at all
    k = torch.zeros(0, 2, 64, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(0, 4, 64, dtype=torch.bfloat16, device="cuda")
    cu = torch.zeros(1, dtype=torch.int32, device="cuda")
    sc, cb = up.score_blocks(q, k, cu, 32, 64)
    keep, kt = up.select_topp(sc, cb, cu, 64, 0.9)
    x = torch.zeros(0, 16, dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros(0, dtype=torch.int32, device="cuda")
    _, _, cuo, tk, _ = up.compact(x, pos, cu, 64, keep, cb)
    torch.cuda.synchronize()
    assert cb.cpu().tolist() == [0] and cuo.cpu().tolist() == [0] and tk.item() == 0


def test_block_larger_than_sequence_and_p_extremes():
    inp = synth.make_inputs([100, 40, 256], 4, 1, 64, 16, 0.05, hidden=32, seed=8)
    full_check(inp, 16, 256, 0.5)           # G >= L: one block per sequence, score 1
    g_sc, g_cb = gpu_scores(inp, 16, 256)
    np.testing.assert_allclose(g_sc, 1.0, atol=1e-5)
    g_sc, g_cb = gpu_scores(inp, 16, 32)
    keep, kt = gpu_select(g_sc, g_cb, inp.cu_seqlens, 32, 1.0)
    assert keep.all() and kt.tolist() == [100, 40, 256]
    keep, kt = gpu_select(g_sc, g_cb, inp.cu_seqlens, 32, 1e-9)
    for s in range(3):
        seg = keep[g_cb[s]:g_cb[s + 1]]
        assert seg.sum() == 1 and np.argmax(seg) == np.argmax(g_sc[g_cb[s]:g_cb[s + 1]])


def _golden_topp():
    out = []
    with open(os.path.join(GOLDEN, "topp_hand_enumerated.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                p, sc, kept = (x.strip() for x in line.split(";"))
                out.append((float(p), [float(v) for v in sc.split(",")],
                            sorted(int(v) for v in kept.split(","))))
    return out


def _golden_topk():
    out = []
    with open(os.path.join(os.path.dirname(__file__), "golden", "topk_hand_enumerated.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, sc, kept = (x.strip() for x in line.split(";"))
                out.append((int(k), [float(v) for v in sc.split(",")],
                            sorted(int(v) for v in kept.split(","))))
    return out


@pytest.mark.parametrize("p,scores,kept", _golden_topp())
def test_select_hand_enumerated(p, scores, kept):
    nb, G = len(scores), 16
    keep, kt = gpu_select(np.array(scores), np.array([0, nb]), np.array([0, nb * G]), G, p)
    assert sorted(np.nonzero(keep)[0].tolist()) == kept
    assert kt.tolist() == [len(kept) * G]


@pytest.mark.parametrize("nb", [1, 2, 1000, 1024, 1025, 4096, 4097, 8192, 16384])
def test_select_ties_and_sizes(nb):
    """Scores with many exact ties (a few distinct values) and all power-of-two
    boundaries of the on-chip sort; the oracle's rule on the same fp32 scores."""
    rng = np.random.default_rng(nb)
    vals = np.array([1.0, 0.5, 0.25, 0.125], dtype=np.float32)
    sc = vals[rng.integers(0, 4, size=nb)].astype(np.float64)
    sc = (sc / sc.sum()).astype(np.float32).astype(np.float64)
    G = 64
    cu = np.array([0, nb * G - 5], np.int32)
    cb = np.array([0, nb], np.int32)
    for p in (0.1, 0.5, 0.9, 0.999, 1.0):
        keep, kt = gpu_select(sc, cb, cu, G, p)
        ok, okt, ci, ce = oracle.select_topp(sc, cb, cu, G, p)
        hard, _ = keep_mismatch(keep, ok, ci, ce, p)
        assert hard == 0
        if np.array_equal(keep, ok):
            assert kt.tolist() == okt.tolist()


def test_select_rejects_too_many_blocks():
    nb = up.SELECT_MAX_BLOCKS + 1
    sc = np.full(nb, 1.0 / nb)
    gpu_select(sc, np.array([0, nb]), np.array([0, nb * 16]), 16, 0.5)
    assert up.get_device_error() == 0x2


@pytest.mark.parametrize("hidden", [8, 520, 4096])
def test_compact_random_keep(hidden):
    rng = np.random.default_rng(hidden)
    lens = [130, 0, 64, 1, 1000, 63]
    G = 32
    cu = np.zeros(len(lens) + 1, np.int32)
    cu[1:] = np.cumsum(lens)
    nbs = [(L + G - 1) // G for L in lens]
    cb = np.zeros(len(lens) + 1, np.int32)
    cb[1:] = np.cumsum(nbs)
    x = rng.integers(0, 1 << 16, size=(int(cu[-1]), hidden), dtype=np.uint16)
    pos = rng.integers(-5, 1 << 30, size=int(cu[-1])).astype(np.int32)
    for prob in (0.0, 0.3, 1.0):
        keep = (rng.random(int(cb[-1])) < prob).astype(np.uint8)
        xo, po, cuo, src, T = gpu_compact(x, pos, cu, G, keep, cb)
        ox, opos, ocu, osrc = oracle.compact(x, pos, cu, G, keep, cb)
        assert T == len(opos)
        np.testing.assert_array_equal(cuo, ocu)
        np.testing.assert_array_equal(src, osrc)
        np.testing.assert_array_equal(po, opos)
        assert np.array_equal(xo, ox)


@pytest.mark.parametrize("G,lens", [
    (32, [130, 0, 64, 1, 1000, 63]),          # one kernel
    (16, [200000, 0, 77, 100003]),            # index kernel + gather (> 16384 blocks)
])
def test_compact_reads_pinned_host_rows_in_place(G, lens):
    """x and pos in pinned host memory: the compaction reads the kept rows in
    place (unified addressing) and gives the oracle's output, bit for bit the
    same as from device copies of x and pos."""
    rng = np.random.default_rng(len(lens))
    cu = np.zeros(len(lens) + 1, np.int32)
    cu[1:] = np.cumsum(lens)
    nbs = [(L + G - 1) // G for L in lens]
    cb = np.zeros(len(lens) + 1, np.int32)
    cb[1:] = np.cumsum(nbs)
    T, hidden = int(cu[-1]), 64
    x_bits = rng.integers(0, 1 << 16, size=(T, hidden), dtype=np.uint16)
    pos = rng.integers(-5, 1 << 30, size=T).astype(np.int32)
    keep = (rng.random(int(cb[-1])) < 0.3).astype(np.uint8)
    x_host = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    pos_host = torch.from_numpy(pos).pin_memory()
    keep_d, cu_d, cb_d = (torch.from_numpy(keep).cuda(), to_dev_i32(cu), to_dev_i32(cb))
    xo, po, cuo, tk, src = up.compact(x_host, pos_host, cu_d, G, keep_d, cb_d)
    xd, pd, _, tkd, _ = up.compact(x_host.cuda(), pos_host.cuda(), cu_d, G, keep_d, cb_d)
    torch.cuda.synchronize()
    n = int(tk.item())
    ox, opos, ocu, osrc = oracle.compact(x_bits, pos, cu, G, keep, cb)
    assert n == len(opos) == int(tkd.item())
    np.testing.assert_array_equal(cuo.cpu().numpy(), ocu)
    np.testing.assert_array_equal(src[:n].cpu().numpy(), osrc)
    np.testing.assert_array_equal(po[:n].cpu().numpy(), opos)
    assert np.array_equal(xo[:n].view(torch.int16).cpu().numpy().view(np.uint16), ox)
    assert torch.equal(xo[:n].view(torch.int16), xd[:n].view(torch.int16))  # bits (NaNs included)
    assert torch.equal(po[:n], pd[:n])
    assert up.get_device_error() == 0


@pytest.mark.parametrize("G,lens,seed", [
    (16, [200000, 0, 77, 100003], 1),       # up to 18759 blocks: index kernel + gather
    (64, [3000] * 300 + [1, 5, 70000], 2),  # 303 sequences, up to 15459 blocks: one kernel
])
def test_compact_both_paths_large_batches(G, lens, seed):
    """Batches on both sides of the one-kernel limit (16384 possible blocks):
    many short sequences and a few long ones, every keep density; bit-exact
    against the oracle."""
    rng = np.random.default_rng(seed)
    cu = np.zeros(len(lens) + 1, np.int32)
    cu[1:] = np.cumsum(lens)
    nbs = [(L + G - 1) // G for L in lens]
    cb = np.zeros(len(lens) + 1, np.int32)
    cb[1:] = np.cumsum(nbs)
    hidden = 8
    x = rng.integers(0, 1 << 16, size=(int(cu[-1]), hidden), dtype=np.uint16)
    pos = rng.integers(-5, 1 << 30, size=int(cu[-1])).astype(np.int32)
    for prob in (0.02, 0.5, 1.0):
        keep = (rng.random(int(cb[-1])) < prob).astype(np.uint8)
        xo, po, cuo, src, T = gpu_compact(x, pos, cu, G, keep, cb)
        ox, opos, ocu, osrc = oracle.compact(x, pos, cu, G, keep, cb)
        assert T == len(opos)
        np.testing.assert_array_equal(cuo, ocu)
        np.testing.assert_array_equal(src, osrc)
        np.testing.assert_array_equal(po, opos)
        assert np.array_equal(xo, ox)


@pytest.mark.parametrize("total", [4096, 2000000])
def test_compact_rejects_a_block_count_the_batch_cannot_have(total):
    """cu_blocks whose last entry exceeds total_tokens/G + num_seqs (here: not
    the cu_blocks of this batch) is caught on the device before any scan or
    scratch write, on both compaction paths: the error bit is set and nothing
    is kept."""
    G = 64
    x = torch.zeros(total, 8, dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros(total, dtype=torch.int32, device="cuda")
    cu = torch.tensor([0, total], dtype=torch.int32, device="cuda")
    bad_nb = total // G + 5
    cb = torch.tensor([0, bad_nb], dtype=torch.int32, device="cuda")
    keep = torch.ones(bad_nb, dtype=torch.uint8, device="cuda")
    _, _, _, tk, _ = up.compact(x, pos, cu, G, keep, cb)
    torch.cuda.synchronize()
    assert int(tk.item()) == 0
    assert up.get_device_error() == 0x10


def test_bad_cu_seqlens_sets_device_error():
    k = torch.zeros(100, 1, 64, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(10, 1, 64, dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 60, 50], dtype=torch.int32, device="cuda")  # decreasing, wrong total
    up.score_blocks(q, k, cu, 5, 64)
    assert up.get_device_error() == 0x1


def test_bad_cu_seqlens_single_sequence():
    """One sequence whose cu_seqlens disagrees with k's length: the scoring
    kernel (which starts from the host's sizes for one sequence) checks the
    bounds itself and loads nothing; the plan reports the error.  q_last holds
    only the rows the given cu_seqlens implies."""
    k = torch.zeros(1000, 1, 64, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(3, 1, 64, dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 3], dtype=torch.int32, device="cuda")  # total should be 1000
    up.score_blocks(q, k, cu, 128, 64)
    torch.cuda.synchronize()
    assert up.get_device_error() == 0x1


# ---------------------------------------------------------------------------
# full-size workloads (the shapes the benchmark times)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name,gain", [
    ("llama31_8b_32k", 5.0),
    ("llama31_8b_128k", 5.0),
    ("llama31_8b_128k", None),
    ("llama31_8b_varlen8_392k", 5.0),
])
def test_full_size_workloads(name, gain):
    w = synth.WORKLOADS[name]
    inp = synth.make_workload(name, gain=gain)
    full_check(inp, w["n"], w["G"], w["p"])


def test_d256_several_units_per_cta():
    """head_dim 256 at 700K tokens: the chunk choice gives 304 units for 152 SMs,
    so every CTA walks two units (the K ring, the Q buffer and the TMEM buffers
    carry over between them, with the per-panel K turnover of head_dim 256)."""
    inp = synth.make_inputs([700000], 8, 1, 256, 128, 0.05, gain=5.0, hidden=64, seed=71)
    full_check(inp, 128, 64, 0.99)


@pytest.mark.parametrize("world", [2, 4])
def test_tensor_parallel_shards_sum_to_all_heads(world):
    """Tensor parallelism simulated on one GPU: each shard of the KV heads (with
    its query heads) is scored with the mean over all query heads; the shards'
    scores sum to the scores of all heads (oracle within the score tolerance),
    each shard's scores sum to its share of the heads per sequence, and
    Hq_total == Hq reproduces score_blocks bit for bit."""
    Hq, Hk, d, n, G = 32, 8, 128, 128, 64
    inp = synth.make_inputs([6000, 2500], Hq, Hk, d, n, 0.05, gain=5.0, hidden=64, seed=29)
    q, k, cu = to_dev_bf16(inp.q_last), to_dev_bf16(inp.k), to_dev_i32(inp.cu_seqlens)
    nb = int(((np.diff(inp.cu_seqlens) + G - 1) // G).sum())
    total = np.zeros(nb)
    cap = inp.total_tokens // G + inp.num_seqs
    for r in range(world):
        qs, ks = up.shard_heads(q, k, r, world)
        # a zero-filled buffer as the all-reduce gets it: the shard call writes
        # only the sum nb_s real entries and leaves the capacity past them at zero
        sc = torch.zeros(cap + 16, dtype=torch.float32, device="cuda")
        sc, cb = up.score_blocks(qs, ks, cu, n, G, scores=sc, Hq_total=Hq)
        torch.cuda.synchronize()
        assert bool((sc[nb:] == 0).all())
        part = sc[:nb].cpu().numpy().astype(np.float64)
        cbn = cb.cpu().numpy()
        for s in range(inp.num_seqs):
            assert abs(part[cbn[s]:cbn[s + 1]].sum() - 1.0 / world) <= 1e-4
        total += part
    orc_sc, orc_cb = oracle.score_blocks(inp.q_last, inp.k, inp.cu_seqlens, Hq, Hk, d, n, G)
    nbad, worst = score_failures(total, orc_sc)
    assert nbad == 0, (nbad, worst)
    full, _ = up.score_blocks(q, k, cu, n, G)
    same, _ = up.score_blocks(q, k, cu, n, G, Hq_total=Hq)
    torch.cuda.synchronize()
    assert torch.equal(full[:nb], same[:nb])


def _paged(inp, page, spare, rng):
    """The token-major keys of a batch cut into pages of `page` tokens at shuffled
    page ids of a pool with `spare` extra pages (filled with other bf16 values);
    unused slots of a sequence's last page hold other values too.
    Returns (k_pages uint16 [P, Hk, page, d], block_table int32 [B, max_pages])."""
    lens = np.diff(inp.cu_seqlens)
    npg = [(int(L) + page - 1) // page for L in lens]
    P = sum(npg) + spare
    Hk, d = inp.Hk, inp.d
    pool = synth.f32_to_bf16_bits(rng.standard_normal((P, Hk, page, d)).astype(np.float32) * 3)
    ids = rng.permutation(P)
    maxp = max(max(npg), 1) + 1
    table = np.full((len(lens), maxp), -1, np.int32)
    nxt = 0
    for s, L in enumerate(lens):
        t0 = int(inp.cu_seqlens[s])
        for i in range(npg[s]):
            pg = int(ids[nxt]); nxt += 1
            table[s, i] = pg
            a, b = i * page, min((i + 1) * page, int(L))
            pool[pg, :, : b - a, :] = inp.k[t0 + a:t0 + b].transpose(1, 0, 2)
    return pool, table


@pytest.mark.parametrize("lens,Hq,Hk,d,page", [
    ([5000], 32, 8, 128, 128),
    ([3000, 0, 1000, 700], 8, 2, 64, 256),
    ([4100], 16, 2, 256, 128),
    ([640, 9000], 32, 8, 128, 384),
])
def test_paged_keys_match_token_major(lens, Hq, Hk, d, page):
    """Keys in a paged, KV-head-major cache (chunked prefill): the scores equal
    those of the same keys laid out token-major bit for bit (same chunks, same
    MMAs; masked slots past a sequence's end hold other values), and the
    oracle's within the tolerance."""
    rng = np.random.default_rng(sum(lens) + page)
    inp = synth.make_inputs(lens, Hq, Hk, d, 128, 0.05, gain=5.0, hidden=64, seed=sum(lens) + 5)
    pool, table = _paged(inp, page, 3, rng)
    q, k, cu = to_dev_bf16(inp.q_last), to_dev_bf16(inp.k), to_dev_i32(inp.cu_seqlens)
    G = 64
    ref, ref_cb = up.score_blocks(q, k, cu, 128, G)
    sc, cb = up.score_blocks_paged(q, to_dev_bf16(pool), torch.from_numpy(table).cuda(), cu,
                                   inp.total_tokens, 128, G)
    torch.cuda.synchronize()
    nb = int(ref_cb[-1].item())
    assert torch.equal(cb, ref_cb)
    assert torch.equal(sc[:nb], ref[:nb])
    orc_sc, _ = oracle.score_blocks(inp.q_last, inp.k, inp.cu_seqlens, Hq, Hk, d, 128, G)
    nbad, worst = score_failures(sc[:nb].cpu().numpy().astype(np.float64), orc_sc)
    assert nbad == 0, (nbad, worst)


def test_paged_keys_bad_page_reads_zeros():
    """A block-table entry past the pool: the error bit is set and that page's
    keys read as zeros (the tensor map bounds the load; nothing faults)."""
    rng = np.random.default_rng(3)
    inp = synth.make_inputs([1000], 8, 2, 64, 32, 0.05, gain=5.0, hidden=64, seed=8)
    pool, table = _paged(inp, 128, 0, rng)
    table[0, 2] = pool.shape[0] + 7
    q, cu = to_dev_bf16(inp.q_last), to_dev_i32(inp.cu_seqlens)
    up.score_blocks_paged(q, to_dev_bf16(pool), torch.from_numpy(table).cuda(), cu,
                          inp.total_tokens, 32, 64)
    torch.cuda.synchronize()
    assert up.get_device_error() == 0x8


@pytest.mark.parametrize("nbs", [[0], [5], [3, 0, 7, 1], [2048], [1000, 0, 2500, 700, 1],
                                 [6272], [300] * 40])
def test_block_csr_matches_oracle(nbs):
    """Block CSR of random keep flags, bit-exact against the oracle: empty
    sequences, fewer blocks than threads, and several blocks per thread."""
    rng = np.random.default_rng(sum(nbs) + len(nbs))
    cb = np.concatenate([[0], np.cumsum(nbs)]).astype(np.int32)
    for frac in (0.0, 0.03, 0.5, 1.0):
        keep = (rng.random(int(cb[-1])) < frac).astype(np.uint8)
        o_ptr, o_idx = oracle.block_csr(keep, cb)
        k_dev = torch.from_numpy(np.concatenate([keep, np.zeros(1, np.uint8)])).cuda()
        ptr, idx = up.block_csr(k_dev, to_dev_i32(cb))
        torch.cuda.synchronize()
        ptr = ptr.cpu().numpy()
        np.testing.assert_array_equal(ptr, o_ptr)
        np.testing.assert_array_equal(idx.cpu().numpy()[: ptr[-1]], o_idx)


def test_full_size_d256_sweep():
    name = "gqa16x2_d256_128k_sweep"
    w = synth.WORKLOADS[name]
    sweep = w["sweep"]
    for n in sweep["n"]:
        inp = synth.make_workload(name, n=n, with_x=(n == 128))
        mass = oracle.token_mass(inp.q_last, inp.k, inp.cu_seqlens, inp.Hq, inp.Hk, inp.d, n)
        for G in sweep["G"]:
            orc_sc, orc_cb = oracle.block_scores(mass, inp.cu_seqlens, G)
            g_sc, g_cb = gpu_scores(inp, n, G)
            np.testing.assert_array_equal(g_cb, orc_cb)
            nbad, worst = score_failures(g_sc, orc_sc)
            assert nbad == 0, (n, G, nbad, worst)
            for p in sweep["p"]:
                ok, _, ci, ce = oracle.select_topp(orc_sc, orc_cb, inp.cu_seqlens, G, p)
                gk, _ = gpu_select(g_sc, g_cb, inp.cu_seqlens, G, p)
                hard, excused = keep_mismatch(gk, ok, ci, ce, p)
                assert hard == 0, (n, G, p, hard)
                if n == 128 and G == 64:
                    xo, po, cuo, src, T = gpu_compact(inp.x, inp.pos, inp.cu_seqlens, G, gk, g_cb)
                    ox, opos, ocu, osrc = oracle.compact(inp.x, inp.pos, inp.cu_seqlens, G, gk, g_cb)
                    assert np.array_equal(xo, ox) and np.array_equal(src, osrc)
                    np.testing.assert_array_equal(cuo, ocu)


def test_overflowing_unit_takes_the_exact_fallback():
    """Among the first 4096 keys of KV head 0, those at positions 100..139 mod 256
    are aligned with the queries' common direction and scaled so their logits
    sit ~130 nats (~190 binary orders) above the other keys.  Work units start
    at multiples of 256 keys, so these keys come after the keys a unit takes its
    reference from; the tensor-core kernel's fp32 sums overflow, and the row
    tiles must be queued and recomputed exactly."""
    inp = synth.make_inputs([32768], 32, 8, 128, 128, 0.05, gain=5.0, hidden=64, seed=11)
    qm = synth.bf16_bits_to_f32(inp.q_last).reshape(-1, 128).mean(axis=0)
    qm /= np.linalg.norm(qm)
    for base in range(0, 4096, 256):
        inp.k[base + 100:base + 140, 0, :] = synth.f32_to_bf16_bits(200.0 * qm)
    q, k, cu = to_dev_bf16(inp.q_last), to_dev_bf16(inp.k), to_dev_i32(inp.cu_seqlens)
    ws = torch.empty(up.score_blocks_workspace(1, 32768, 32, 8, 128, 128, 64),
                     dtype=torch.uint8, device="cuda")
    sc, cb = up.score_blocks(q, k, cu, 128, 64, workspace=ws)
    torch.cuda.synchronize()
    flagged = int(ws[256 + 16:256 + 20].view(torch.int32).item())
    assert flagged > 0, "the overflowing unit was not queued for the fallback"
    # with a queue, every CTA of the scoring kernel recomputes its share of the
    # queued tiles and then arrives at the fallback's grid barrier
    fallback_barrier = int(ws[256 + 28:256 + 32].view(torch.int32).item())
    assert fallback_barrier > 0
    orc_sc, orc_cb = oracle.score_blocks(inp.q_last, inp.k, inp.cu_seqlens, 32, 8, 128, 128, 64)
    g_sc = sc[: int(orc_cb[-1])].cpu().numpy().astype(np.float64)
    nbad, worst = score_failures(g_sc, orc_sc)
    assert nbad == 0, (nbad, worst)
    assert up.get_device_error() == 0
    # the same keys in a paged cache: the fallback reads them through the block table
    pool, table = _paged(inp, 256, 2, np.random.default_rng(4))
    ws.zero_()
    psc, _ = up.score_blocks_paged(q, to_dev_bf16(pool), torch.from_numpy(table).cuda(), cu,
                                   32768, 128, 64, workspace=ws)
    torch.cuda.synchronize()
    assert int(ws[256 + 16:256 + 20].view(torch.int32).item()) > 0
    assert torch.equal(psc[: int(orc_cb[-1])], sc[: int(orc_cb[-1])])
    assert up.get_device_error() == 0


def test_expired_wait_stops_the_scoring_kernel_cleanly():
    """Failure detection without a fault: with the spin-wait bound lowered to a
    few hundred cycles, the scoring kernel's first waits for data run out.
    The call still returns, every CTA stops (copies and MMAs in flight are
    drained, tensor memory freed), the timeout bit reaches the host through
    the device error word, and the next call at the default bound matches the
    oracle on the same context."""
    inp = synth.make_inputs([6000, 3000], 8, 2, 128, 128, 0.05, gain=5.0, hidden=64, seed=21)
    q, k, cu = to_dev_bf16(inp.q_last), to_dev_bf16(inp.k), to_dev_i32(inp.cu_seqlens)
    assert up.get_device_error() == 0
    up.set_wait_limit(300)
    try:
        up.score_blocks(q, k, cu, 128, 64)
        torch.cuda.synchronize()
    finally:
        up.set_wait_limit(0)
    bits = up.get_device_error()
    assert bits & 0x4, f"the timeout bit was not set (bits {bits:#x})"
    full_check(inp, 128, 64, 0.99)
    assert up.get_device_error() == 0


@pytest.mark.gpu
def test_ex2_rate_probe():
    """The exponential-roof microbenchmark returns a plausible device-wide rate
    (a GB300 runs tens of ex2 per clock per SM on 152 SMs at ~2 GHz)."""
    rate = up.measure_ex2_rate()
    assert 1e11 < rate < 1e15


def gpu_select_blocks(scores_np, cb_np, cu_np, G, **kw):
    sc = torch.from_numpy(np.ascontiguousarray(scores_np, dtype=np.float32)).cuda()
    keep, kt = up.select_blocks(sc, torch.from_numpy(np.ascontiguousarray(cb_np, np.int32)).cuda(),
                                torch.from_numpy(np.ascontiguousarray(cu_np, np.int32)).cuda(), G, **kw)
    torch.cuda.synchronize()
    return keep[: len(scores_np)].cpu().numpy(), kt[: len(cu_np) - 1].cpu().numpy()


@pytest.mark.gpu
@pytest.mark.parametrize("k,scores,kept", _golden_topk())
def test_select_topk_hand_enumerated(k, scores, kept):
    nb, G = len(scores), 16
    keep, kt = gpu_select_blocks(np.array(scores), np.array([0, nb]), np.array([0, nb * G]), G,
                                 mode="top_k", k=k)
    assert sorted(np.nonzero(keep)[0].tolist()) == kept
    assert kt.tolist() == [len(kept) * G]


@pytest.mark.gpu
@pytest.mark.parametrize("nb", [1, 2, 513, 1024, 1025, 4096, 4097, 8192, 16384])
def test_select_topk_ties_and_sizes(nb):
    """Top-k on scores with many exact ties, at every power-of-two size boundary of
    the kernel, against the oracle on the same fp32 scores (unique result)."""
    rng = np.random.default_rng(nb + 7)
    vals = np.array([1.0, 0.5, 0.25, 0.125], dtype=np.float32)
    sc = vals[rng.integers(0, 4, size=nb)].astype(np.float64)
    sc = (sc / sc.sum()).astype(np.float32).astype(np.float64)
    G = 64
    cu = np.array([0, nb * G - 5], np.int32)
    cb = np.array([0, nb], np.int32)
    for k in sorted({1, 2, max(1, nb // 3), nb - 1 if nb > 1 else 1, nb, nb + 5}):
        keep, kt = gpu_select_blocks(sc, cb, cu, G, mode="top_k", k=k)
        ok, okt = oracle.select_topk(sc, cb, cu, G, k)
        np.testing.assert_array_equal(keep, ok)
        assert kt.tolist() == okt.tolist()


@pytest.mark.gpu
def test_select_topp_varlen_both_paths():
    """Top-p on a varlen batch whose sequences take both selection paths: up to
    4096 blocks the per-block exact mass-before over many CTAs, above it the
    one-CTA radix search (ragged last blocks, an empty sequence)."""
    rng = np.random.default_rng(23)
    G = 64
    lens = [64 * 5000 + 17, 300, 0, 64 * 4096, 64 * 4097 - 3, 64 * 2048]
    cu = np.array([0] + list(np.cumsum(lens)), np.int32)
    nbs = [(L + G - 1) // G for L in lens]
    cb = np.array([0] + list(np.cumsum(nbs)), np.int32)
    parts = []
    for nb in nbs:
        r = rng.exponential(size=nb) ** 3
        parts.append(r / r.sum() if nb else r)
    sc = np.concatenate(parts).astype(np.float32).astype(np.float64)
    for p in (0.5, 0.9, 0.99):
        keep, kt = gpu_select(sc, cb, cu, G, p)
        ok, okt, ci, ce = oracle.select_topp(sc, cb, cu, G, p)
        hard, _ = keep_mismatch(keep, ok, ci, ce, p)
        assert hard == 0
        if np.array_equal(keep, ok):
            assert kt.tolist() == okt.tolist()


@pytest.mark.gpu
def test_select_topk_varlen_random_scores():
    """Varlen batch (including an empty sequence) of continuous random scores."""
    rng = np.random.default_rng(11)
    lens = [640, 0, 4100, 64, 131072]
    G = 64
    cu = np.array([0] + list(np.cumsum(lens)), np.int32)
    nbs = [(L + G - 1) // G for L in lens]
    cb = np.array([0] + list(np.cumsum(nbs)), np.int32)
    parts = []
    for nb in nbs:
        r = rng.exponential(size=nb) ** 2
        parts.append(r / r.sum() if nb else r)
    sc = np.concatenate(parts).astype(np.float32).astype(np.float64)
    for k in (1, 5, 41, 3000):
        keep, kt = gpu_select_blocks(sc, cb, cu, G, mode="top_k", k=k)
        ok, okt = oracle.select_topk(sc, cb, cu, G, k)
        np.testing.assert_array_equal(keep, ok)
        assert kt.tolist() == okt.tolist()


@pytest.mark.gpu
@pytest.mark.parametrize("mode", ["top_p", "top_k"])
def test_select_keep_last_option(mode):
    """The keep-last flag equals the oracle's selection followed by its keep-last
    step, for both rules, on a varlen batch with ragged last blocks."""
    rng = np.random.default_rng(5)
    lens = [1000, 37, 0, 5000, 64]
    G = 64
    cu = np.array([0] + list(np.cumsum(lens)), np.int32)
    nbs = [(L + G - 1) // G for L in lens]
    cb = np.array([0] + list(np.cumsum(nbs)), np.int32)
    parts = []
    for nb in nbs:
        r = rng.exponential(size=nb) ** 3
        parts.append(r / r.sum() if nb else r)
    sc = np.concatenate(parts).astype(np.float32).astype(np.float64)
    if mode == "top_p":
        keep, kt = gpu_select_blocks(sc, cb, cu, G, mode="top_p", p=0.9, keep_last=True)
        ok, okt, ci, ce = oracle.select_topp(sc, cb, cu, G, 0.9)
        hard, _ = keep_mismatch(keep, oracle.keep_last_block(ok, okt, cb, cu, G)[0], ci, ce, 0.9)
        assert hard == 0
        ok2, okt2 = oracle.keep_last_block(ok, okt, cb, cu, G)
        if np.array_equal(keep, ok2):
            assert kt.tolist() == okt2.tolist()
    else:
        keep, kt = gpu_select_blocks(sc, cb, cu, G, mode="top_k", k=3, keep_last=True)
        ok, okt = oracle.select_topk(sc, cb, cu, G, 3)
        ok2, okt2 = oracle.keep_last_block(ok, okt, cb, cu, G)
        np.testing.assert_array_equal(keep, ok2)
        assert kt.tolist() == okt2.tolist()
    # every non-empty sequence keeps its last block
    for s in range(len(lens)):
        if nbs[s]:
            assert keep[cb[s + 1] - 1] == 1


def test_checked_build_matches_the_oracle_with_no_bounds_miss(monkeypatch):
    """The checked build (-DUP_CHECK_BOUNDS: every kernel tests the index ranges
    it reads and writes, and reports a miss through UP_DEVERR_BOUNDS instead of
    trapping) runs the whole path on shapes chosen for their edges -- ragged
    tiles and blocks, empty and one-token sequences, every head_dim, G = 16
    and 256, paged keys, the compaction's index + gather path -- and must give
    the oracle's results with no error bit set."""
    checked = up.load_library(up._build.build(checked=True))
    monkeypatch.setattr(up, "_lib", checked)
    assert up.get_device_error() == 0
    for lens, Hq, Hk, d, n, G, p in [
            ([300, 129, 4100], 4, 1, 64, 16, 256, 0.9),
            ([5, 1, 0, 129], 4, 4, 64, 128, 32, 0.99),
            ([9000], 12, 4, 128, 48, 16, 0.999),
            ([2048], 16, 2, 256, 100, 128, 0.9)]:
        inp = synth.make_inputs(lens, Hq, Hk, d, n, 0.05, gain=5.0, hidden=64,
                                seed=sum(lens) + d)
        full_check(inp, n, G, p)
        assert up.get_device_error() == 0, (lens, d, G)
    # paged keys
    inp = synth.make_inputs([3000, 700], 8, 2, 128, 64, 0.05, gain=5.0, hidden=64, seed=5)
    pool, table = _paged(inp, 256, 3, np.random.default_rng(6))
    q, cu = to_dev_bf16(inp.q_last), to_dev_i32(inp.cu_seqlens)
    psc, pcb = up.score_blocks_paged(q, to_dev_bf16(pool), torch.from_numpy(table).cuda(), cu,
                                     inp.total_tokens, 64, 64)
    sc, cb = up.score_blocks(q, to_dev_bf16(inp.k), cu, 64, 64)
    torch.cuda.synchronize()
    assert torch.equal(psc[: int(cb[-1])], sc[: int(cb[-1])])
    assert up.get_device_error() == 0
    # the compaction's two-kernel path (more than 16384 possible blocks)
    G, lens = 16, [200000, 0, 77, 100003]
    rng = np.random.default_rng(9)
    cu_np = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cb_np = np.concatenate([[0], np.cumsum([(L + G - 1) // G for L in lens])]).astype(np.int32)
    x = rng.integers(0, 1 << 16, size=(int(cu_np[-1]), 8), dtype=np.uint16)
    pos = np.arange(int(cu_np[-1]), dtype=np.int32)
    keep = (rng.random(int(cb_np[-1])) < 0.3).astype(np.uint8)
    xo, po, cuo, src, T = gpu_compact(x, pos, cu_np, G, keep, cb_np)
    ox, opos, ocu, osrc = oracle.compact(x, pos, cu_np, G, keep, cb_np)
    assert T == len(opos) and np.array_equal(xo, ox)
    np.testing.assert_array_equal(src, osrc)
    assert up.get_device_error() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("nb", [40, 1500, 4096])
def test_select_threshold_filter_edges(nb):
    """Scores placed at and around the selection's filter thresholds (2^-8,
    2^-14, 2^-20: exact binary values, their neighbours and the ranges between)
    with p chosen so that each threshold, or none, is the highest whose keys at
    or above hold p; top-p and top-k against the oracle on the same fp32 scores."""
    rng = np.random.default_rng(nb)
    edges = []
    for j in (8, 14, 20):
        t = np.float32(2.0 ** -j)
        edges += [t, np.nextafter(t, np.float32(1)), np.nextafter(t, np.float32(0))]
    sc = np.concatenate([np.array(edges, np.float32),
                         np.float32(2.0) ** -rng.uniform(0, 26, size=nb - len(edges)).astype(np.float32)])
    sc = rng.permutation(sc / sc.sum()).astype(np.float32).astype(np.float64)
    G = 64
    cu = np.array([0, nb * G - 3], np.int32)
    cb = np.array([0, nb], np.int32)
    order = np.sort(sc)[::-1]
    ps = {0.3, 0.9, 0.999, 1.0}
    for j in (8, 14, 20):  # p right at, just above and just below each threshold's own mass
        at = float(order[order >= 2.0 ** -j].sum())
        ps |= {min(at, 1.0), min(np.nextafter(at, 2.0), 1.0), np.nextafter(at, 0.0)}
    for p in sorted(x for x in ps if x > 0):
        keep, kt = gpu_select(sc, cb, cu, G, p)
        ok, okt, ci, ce = oracle.select_topp(sc, cb, cu, G, p)
        hard, _ = keep_mismatch(keep, ok, ci, ce, p)
        assert hard == 0, (nb, p)
    for k in sorted({1, 3, len(edges), nb // 2, nb - 1}):
        keep, kt = gpu_select_blocks(sc, cb, cu, G, mode="top_k", k=k)
        ok, okt = oracle.select_topk(sc, cb, cu, G, k)
        np.testing.assert_array_equal(keep, ok)
        np.testing.assert_array_equal(kt, okt)
    assert up.get_device_error() == 0
