"""The multi-process (N > 1) paths of bench.py, exercised with gloo on CPU.

The hot path shards by sequence with no data-path collective; N ranks run N
replicas and bench.py takes the max over ranks of the step time.  These tests
cover the host-side rank logic: the max-over-ranks reduction and the reference
arm under torchrun (rank 0 alone prints one JSON line, other ranks exit 0).
The tensor-parallel mode (heads sharded over ranks, block scores summed by an
all-reduce) is covered with CPU ranks whose per-shard scores come from the
oracle under the library's shard contract.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w = bench.dist_setup()
    assert (r, w) == (rank, world)
    bench.barrier(w)
    out[rank] = bench.max_over_ranks(float(rank + 1) * 1.5, w)
    torch.distributed.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        assert dict(out) == {0: 3.0, 1: 3.0}


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "2", "--warmup", "1", "--workload",
           "gqa8x2_d64_4k"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["config"]["workload"] == "gqa8x2_d64_4k"


def _tp_rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import numpy as np
    import torch.distributed as dist
    import block_sparse_long_up_gb300 as up
    import oracle
    from block_sparse_long_up_gb300 import synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    Hq, Hk, d, n, G = 8, 4, 64, 32, 16
    inp = synth.make_inputs([700, 0, 300], Hq, Hk, d, n, 0.05, gain=5.0, hidden=8, seed=3)
    as_bf16 = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
        torch.bfloat16)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    q, k = as_bf16(inp.q_last), as_bf16(inp.k)
    cu = torch.from_numpy(inp.cu_seqlens)

    def shard_contract(q_last, k_sh, cu_seqlens, n_, G_, scores=None, stream=None,
                       Hq_total=None):
        # up_score_blocks_shard's definition: this shard's heads, mean over Hq_total,
        # written into the caller's buffer (whose capacity past sum nb_s stays as given)
        sc, cb = oracle.score_blocks(bits(q_last), bits(k_sh), cu_seqlens.numpy(),
                                     q_last.shape[1], k_sh.shape[1], d, n_, G_)
        out = scores.to(torch.float64)
        out[:len(sc)] = torch.from_numpy(sc * (q_last.shape[1] / Hq_total))
        return out, torch.from_numpy(cb)

    up.score_blocks = shard_contract  # tp_score_blocks calls the module's score_blocks
    qs, ks = up.shard_heads(q, k, rank, world)
    assert qs.shape[1] == Hq // world and ks.shape[1] == Hk // world
    sc, cb = up.tp_score_blocks(qs, ks, cu, n, G, Hq)
    full, fcb = oracle.score_blocks(inp.q_last, inp.k, inp.cu_seqlens, Hq, Hk, d, n, G)
    assert np.array_equal(cb.numpy(), fcb)
    nb = len(full)
    assert float(sc[nb:].abs().sum()) == 0.0  # the zeroed capacity stays zero after the sum
    out[rank] = float(np.max(np.abs(sc[:nb].numpy() - full)))
    dist.destroy_process_group()


def test_tensor_parallel_scores_gloo_two_ranks():
    """Two ranks each hold half of the KV heads (and their query heads); their
    shard scores, summed by the all-reduce, equal the scores of all heads."""
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_tp_rank_main, args=(2, port, out), nprocs=2, join=True)
        assert set(out.keys()) == {0, 1}
        assert max(out.values()) < 1e-12, dict(out)
