"""Seeded synthetic inputs for block scoring, top-p selection and compaction.

This module only draws random numbers; it holds none of the method's
arithmetic.  Both the CUDA path and the CPU oracle read the same bits from it.

Recipe (the UniPrefill pages evaluate Llama-3.1-8B on RULER at 128K; no model
weights or dataset are used here -- these shapes and distributions stand in):

* q_last, k: i.i.d. N(0, 1) per coordinate, drawn in fp32 from numpy's PCG64
  (one SeedSequence child stream per tensor), shifted, then rounded to bf16
  with round-to-nearest-even.
* u: one N(0, I_d) vector normalised to unit length, shared by all heads.
* sink: every key of block 0 (blocks of ``plant_block`` = 64 tokens) gets
  +3*s*u; salient: round(f*(nb-1)) blocks drawn without replacement from
  1..nb-1 get +2*s*u on their keys; every query row of every head gets +1*s*u.
* s = 1 is the literal reading of a unit-vector shift.  That barely moves the
  logits (3/sqrt(d)), so nearly every block survives top-p.  The "gain"
  reading s = sqrt(lam)*d**0.25 turns the shifts into logit offsets of
  3*lam / 2*lam (+15 / +10 at lam = 5) at every head_dim, which gives the low
  retention ratio the long-context workloads call for.
* x: N(0, 1) bf16 [total_tokens, hidden]; pos: int32 0..L_s-1 per sequence.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

PLANT_BLOCK = 64


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest-even) and return the uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def shift_scale(d: int, gain) -> float:
    """s for a head_dim d: 1 for the literal reading, sqrt(gain)*d**0.25 otherwise."""
    if gain is None:
        return 1.0
    return math.sqrt(float(gain)) * float(d) ** 0.25


@dataclasses.dataclass
class Inputs:
    q_last: np.ndarray      # uint16 [sum n_s, Hq, d]
    k: np.ndarray           # uint16 [total, Hk, d]
    cu_seqlens: np.ndarray  # int32 [B+1]
    x: np.ndarray | None    # uint16 [total, hidden]
    pos: np.ndarray         # int32 [total]
    Hq: int
    Hk: int
    d: int
    n: int
    hidden: int
    salient: list           # per-sequence salient fraction
    gain: float | None
    planted: list = dataclasses.field(default_factory=list)  # per sequence: salient planting blocks

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def num_seqs(self) -> int:
        return int(self.cu_seqlens.shape[0] - 1)


def _normal_bf16(rng: np.random.Generator, shape, shift_rows=None, chunk=1 << 26):
    """N(0,1) bf16 bits of the given shape; ``shift_rows(first_row, block)`` may add a shift."""
    out = np.empty(shape, dtype=np.uint16)
    flat_rows = out.reshape(shape[0], -1)
    row_elems = flat_rows.shape[1]
    rows_per_chunk = max(1, chunk // max(1, row_elems))
    for r0 in range(0, shape[0], rows_per_chunk):
        r1 = min(shape[0], r0 + rows_per_chunk)
        v = rng.standard_normal((r1 - r0,) + tuple(shape[1:]), dtype=np.float32)
        if shift_rows is not None:
            shift_rows(r0, v)
        flat_rows[r0:r1] = f32_to_bf16_bits(v).reshape(r1 - r0, -1)
    return out


def make_inputs(lens, Hq, Hk, d, n, salient, gain=5.0, hidden=None, seed=1000,
                with_x=True, plant_block=PLANT_BLOCK) -> Inputs:
    """Draw one varlen batch.

    lens: sequence lengths; salient: one fraction for all sequences, or a
    (lo, hi) tuple to draw each sequence's fraction uniformly from; gain: None
    for the literal unit shift, else the logit gain described above.
    """
    lens = [int(v) for v in lens]
    B = len(lens)
    ss = np.random.SeedSequence(seed)
    s_u, s_sal, s_q, s_k, s_x = ss.spawn(5)
    rng_u = np.random.Generator(np.random.PCG64(s_u))
    u = rng_u.standard_normal(d)
    u = (u / np.linalg.norm(u)).astype(np.float32)
    s = np.float32(shift_scale(d, gain))

    rng_sal = np.random.Generator(np.random.PCG64(s_sal))
    if isinstance(salient, tuple):
        fracs = [float(rng_sal.uniform(salient[0], salient[1])) for _ in range(B)]
    else:
        fracs = [float(salient)] * B
    plant = []
    for L, f in zip(lens, fracs):
        nbp = (L + plant_block - 1) // plant_block
        m = int(round(f * (nbp - 1)))
        chosen = rng_sal.choice(np.arange(1, nbp), size=m, replace=False) if m > 0 else np.zeros(0, np.int64)
        plant.append(np.sort(chosen))

    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    total = int(cu[-1])

    # keys: one stream, sequence after sequence
    rng_k = np.random.Generator(np.random.PCG64(s_k))
    k = np.empty((total, Hk, d), dtype=np.uint16)
    for si, L in enumerate(lens):
        if L == 0:
            continue
        mult = np.zeros((L + plant_block - 1) // plant_block, dtype=np.float32)
        mult[0] = 3.0
        mult[plant[si]] = 2.0

        def shift(r0, v, mult=mult):
            rows = np.arange(r0, r0 + v.shape[0]) // plant_block
            v += (mult[rows] * s)[:, None, None] * u[None, None, :]

        k[cu[si]:cu[si + 1]] = _normal_bf16(rng_k, (L, Hk, d), shift)

    nq = [min(n, L) for L in lens]
    rng_q = np.random.Generator(np.random.PCG64(s_q))
    qv = rng_q.standard_normal((sum(nq), Hq, d), dtype=np.float32)
    qv += s * u[None, None, :]
    q_last = f32_to_bf16_bits(qv)

    x = None
    if with_x and hidden:
        rng_x = np.random.Generator(np.random.PCG64(s_x))
        x = _normal_bf16(rng_x, (total, hidden))
    pos = np.concatenate([np.arange(L, dtype=np.int32) for L in lens]) if total else np.zeros(0, np.int32)
    return Inputs(q_last=q_last, k=k, cu_seqlens=cu, x=x, pos=pos, Hq=Hq, Hk=Hk, d=d, n=n,
                  hidden=int(hidden or 0), salient=fracs, gain=gain, planted=plant)


# Named workloads (shapes from the long-context prefill setting the pages
# evaluate: Llama-3.1-8B layers at up to 128K tokens, plus a small GQA case and
# a head_dim-256 sweep layer).
WORKLOADS = {
    "gqa8x2_d64_4k": dict(lens=[4096], Hq=8, Hk=2, d=64, hidden=512, n=128, G=64, p=0.99,
                          salient=0.05, seed=1001),
    "llama31_8b_32k": dict(lens=[32768], Hq=32, Hk=8, d=128, hidden=4096, n=128, G=64, p=0.99,
                           salient=0.05, seed=1002),
    "llama31_8b_128k": dict(lens=[131072], Hq=32, Hk=8, d=128, hidden=4096, n=128, G=64, p=0.99,
                            salient=0.02, seed=1003),
    "llama31_8b_varlen8_392k": dict(lens=[8192, 16384, 16384, 32768, 32768, 65536, 98304, 131072],
                                    Hq=32, Hk=8, d=128, hidden=4096, n=128, G=64, p=0.99,
                                    salient=(0.01, 0.10), seed=1004),
    "gqa16x2_d256_128k_sweep": dict(lens=[131072], Hq=16, Hk=2, d=256, hidden=2048, n=128, G=64,
                                    p=0.99, salient=0.05, seed=1005,
                                    sweep=dict(p=[0.9, 0.95, 0.99, 0.999], G=[32, 64, 128],
                                               n=[64, 128, 256])),
}


def make_workload(name, gain=5.0, with_x=True, n=None, lens=None, seed=None) -> Inputs:
    w = WORKLOADS[name]
    return make_inputs(lens if lens is not None else w["lens"], w["Hq"], w["Hk"], w["d"],
                       n if n is not None else w["n"], w["salient"], gain=gain,
                       hidden=w["hidden"], seed=w["seed"] if seed is None else seed,
                       with_x=with_x)
