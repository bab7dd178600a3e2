"""The C-ABI library builds, loads without a GPU, exports what include/up.h
declares, and rejects bad host-side arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

import block_sparse_long_up_gb300 as up

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    up.build()
    return up.lib()


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(up_[a-z0-9_]+)\s*\(", text))
    return names


def test_header_is_plain_c(tmp_path):
    """include/up.h compiles as C99 with warnings as errors, and every declared
    entry point can be named from C (its address taken), so a C caller needs
    nothing but the header and the shared library."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = sorted(_declared_functions())
    src = tmp_path / "use_up.c"
    src.write_text('#include "up.h"\n'
                   "typedef void (*up_fn)(void);\n"
                   "up_fn up_entry_points[] = {\n" +
                   "".join(f"    (up_fn)&{n},\n" for n in names) + "};\n")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic-errors",
                        "-I", os.path.join(ROOT, "include"), "-c", str(src),
                        "-o", str(tmp_path / "use_up.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_exports_every_declared_symbol(L):
    names = _declared_functions()
    assert {"up_score_blocks", "up_select_topp", "up_compact"} <= names
    for name in sorted(names):
        assert hasattr(L, name), f"{name} is declared in include/ but not exported"


def test_status_strings(L):
    for code in range(7):
        assert L.up_status_string(code)
    assert L.up_status_string(0) == b"ok"


def test_workspace_sizes(L):
    # the Llama-3.1-8B layer at 128K: partial sums of 4096 rows x 2048 blocks dominate
    ws = up.score_blocks_workspace(1, 131072, 32, 8, 128, 128, 64)
    assert 4096 * 2049 * 4 <= ws < 64 << 20
    assert up.score_blocks_workspace(1, 4096, 8, 2, 64, 128, 64) > 0
    # unsupported shapes report 0
    assert up.score_blocks_workspace(1, 4096, 8, 3, 64, 128, 64) == 0
    assert up.score_blocks_workspace(1, 4096, 8, 2, 96, 128, 64) == 0
    assert up.score_blocks_workspace(1, 4096, 8, 2, 64, 128, 48) == 0
    assert up.compact_workspace(8, 401408, 64) >= (401408 // 64 + 8) * 20
    assert up.compact_workspace(1, 100, 7) == 0


P = ctypes.c_void_p


def _fake(addr=256):
    return ctypes.c_void_p(addr)


def test_score_rejects_bad_arguments(L):
    args = dict(q=_fake(), k=_fake(), cu=_fake(), B=1, T=4096, Hq=8, Hk=2, d=64, n=128, G=64,
                sc=_fake(), cb=_fake(), ws=_fake(), wsb=1 << 30)

    def call(**kw):
        a = dict(args, **kw)
        return L.up_score_blocks(a["q"], a["k"], a["cu"], a["B"], a["T"], a["Hq"], a["Hk"],
                                 a["d"], a["n"], a["G"], a["sc"], a["cb"], a["ws"], a["wsb"], None)

    assert call(Hk=3) == 1          # Hq % Hk
    assert call(n=0) == 1
    assert call(B=-1) == 1
    assert call(cu=None) == 1
    assert call(q=None) == 1
    assert call(q=_fake(258)) == 1  # q_last not 16-byte aligned
    assert call(d=96) == 2
    assert call(G=48) == 2
    assert call(n=2048) == 2
    assert call(Hq=64, Hk=2) == 2   # group of 32 query heads per KV head
    assert call(ws=None) == 3
    assert call(wsb=1024) == 3
    assert call(ws=_fake(272)) == 3  # workspace not 256-byte aligned


def test_score_shard_rejects_too_few_total_heads(L):
    # Hq_total below the shard's own query heads
    assert L.up_score_blocks_shard(_fake(), _fake(), _fake(), 1, 4096, 8, 2, 64, 128, 64, 4,
                                   _fake(), _fake(), _fake(), 1 << 30, None) == 1
    assert L.up_score_blocks_shard(_fake(), _fake(), _fake(), 1, 4096, 8, 2, 64, 128, 64, 0,
                                   _fake(), _fake(), _fake(), 1 << 30, None) == 1


def test_score_paged_rejects_bad_arguments(L):
    def call(pages=64, page=128, table=_fake(), maxp=8, B=2, T=4096):
        return L.up_score_blocks_paged(_fake(), _fake(), pages, page, table, maxp, _fake(), B, T,
                                       8, 2, 64, 128, 64, _fake(), _fake(), _fake(), 1 << 30, None)

    assert call(table=None) == 1
    assert call(page=64) == 1           # not a multiple of 128
    assert call(page=200) == 1
    assert call(pages=0) == 1
    assert call(maxp=0) == 1
    assert call(pages=1 << 22, page=1024) == 1   # rows past 2^31
    assert call(B=1, T=4096, maxp=31) == 1       # one sequence longer than its table row


def test_block_csr_rejects_bad_arguments(L):
    assert L.up_block_csr(None, _fake(), 1, _fake(), _fake(), None) == 1
    assert L.up_block_csr(_fake(), None, 1, _fake(), _fake(), None) == 1
    assert L.up_block_csr(_fake(), _fake(), 1, None, _fake(), None) == 1
    assert L.up_block_csr(_fake(), _fake(), 1, _fake(), None, None) == 1
    assert L.up_block_csr(_fake(), _fake(), -1, _fake(), _fake(), None) == 1


def test_select_and_compact_reject_bad_arguments(L):
    assert L.up_select_topp(_fake(), _fake(), _fake(), 1, 64, 0.0, _fake(), _fake(), None) == 1
    assert L.up_select_topp(_fake(), _fake(), _fake(), 1, 64, float("nan"), _fake(), _fake(), None) == 1
    assert L.up_select_topp(_fake(), _fake(), _fake(), 1, 40, 0.9, _fake(), _fake(), None) == 2
    assert L.up_select_topp(None, _fake(), _fake(), 1, 64, 0.9, _fake(), _fake(), None) == 1

    def sel(mode=0, p=0.9, k=4, flags=0, G=64, sc=_fake()):
        return L.up_select_blocks(sc, _fake(), _fake(), 1, G, mode, p, k, flags, _fake(), _fake(),
                                  None)

    assert sel(mode=2) == 1              # unknown mode
    assert sel(flags=0x2) == 1           # unknown flag bit
    assert sel(mode=0, p=0.0) == 1
    assert sel(mode=0, p=float("nan")) == 1
    assert sel(mode=1, k=0) == 1
    assert sel(mode=1, G=40) == 2
    assert sel(mode=1, sc=None) == 1

    def comp(hidden=512, x=_fake(), xo=_fake(), ws=_fake(), wsb=1 << 30, G=64, tk=_fake()):
        return L.up_compact(x, _fake(), hidden, _fake(), 1, 4096, G, _fake(), _fake(), xo,
                            _fake(), _fake(), None, tk, ws, wsb, None)

    assert comp(hidden=500) == 2
    assert comp(G=65) == 2
    assert comp(x=_fake(264)) == 1
    assert comp(xo=_fake(264)) == 1
    assert comp(tk=None) == 1
    assert comp(ws=None) == 3
    assert comp(wsb=16) == 3


def test_python_binding_fails_loudly_without_cuda_tensors(L):
    import torch
    q = torch.zeros(4, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        up.score_blocks(q, q, torch.zeros(2, dtype=torch.int32), 4, 64)


def test_oracle_and_kernels_share_no_code():
    """The oracle (plain C, test infrastructure) and the CUDA library include
    nothing from each other, and the product package never imports the oracle:
    there is no CPU path behind the library's calls."""
    pkg = os.path.join(ROOT, "block_sparse_long_up_gb300")
    csrc = os.path.join(pkg, "csrc")
    for fn in os.listdir(csrc):
        text = open(os.path.join(csrc, fn)).read()
        assert "oracle" not in text.lower(), fn
    for fn in os.listdir(os.path.join(ROOT, "oracle")):
        if fn.endswith((".c", ".h", ".py")):
            text = open(os.path.join(ROOT, "oracle", fn)).read()
            assert "csrc" not in text and "up.h" not in text and "block_sparse_long_up_gb300" not in text, fn
    for fn in os.listdir(pkg):
        if fn.endswith(".py"):
            text = open(os.path.join(pkg, fn)).read()
            assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), fn


def test_wait_limit_bounds(L):
    """The failure-path hook takes a bound up to the default and 0 (restore)."""
    assert L.up_set_wait_limit(ctypes.c_uint64(1 << 62)) == 1
    assert L.up_set_wait_limit(ctypes.c_uint64(5000)) == 0
    assert L.up_set_wait_limit(ctypes.c_uint64(0)) == 0


def test_compact_noalloc_checks_every_tensor_before_the_library(monkeypatch):
    """Every argument of the no-workspace compaction is checked in Python
    (type, dtype, size, then device) before anything reaches the C library: a
    wrong dtype that would make the kernel read or write out of bounds raises
    first."""
    import torch

    def no_library():
        raise AssertionError("the C library was reached")

    monkeypatch.setattr(up, "lib", no_library)
    T, H, G, B = 256, 16, 64, 2
    good = dict(x=torch.zeros(T, H, dtype=torch.bfloat16), pos=torch.zeros(T, dtype=torch.int32),
                cu_seqlens=torch.tensor([0, 100, T], dtype=torch.int32), G=G,
                keep=torch.zeros(T // G + B, dtype=torch.uint8),
                cu_blocks=torch.zeros(B + 1, dtype=torch.int32),
                x_out=torch.zeros(T, H, dtype=torch.bfloat16),
                pos_out=torch.zeros(T, dtype=torch.int32),
                cu_seqlens_out=torch.zeros(B + 1, dtype=torch.int32),
                src_idx=torch.zeros(T, dtype=torch.int32),
                total_kept=torch.zeros(1, dtype=torch.int32))
    wrong_dtype = dict(keep=torch.int64, pos=torch.float32, cu_seqlens=torch.int64,
                       cu_blocks=torch.int64, x_out=torch.float16, pos_out=torch.int64,
                       cu_seqlens_out=torch.int16, src_idx=torch.int64, total_kept=torch.int64,
                       x=torch.float32)
    for name, dt in wrong_dtype.items():
        args = dict(good)
        args[name] = args[name].to(dt)
        with pytest.raises(TypeError, match=name):
            up.compact_noalloc(**args)
    for name, short in (("pos_out", torch.zeros(T - 1, dtype=torch.int32)),
                        ("src_idx", torch.zeros(T - 1, dtype=torch.int32)),
                        ("cu_blocks", torch.zeros(B, dtype=torch.int32))):
        args = dict(good)
        args[name] = short
        with pytest.raises(ValueError):
            up.compact_noalloc(**args)
    with pytest.raises(ValueError, match="CUDA"):
        up.compact_noalloc(**good)  # right dtypes and sizes, but host tensors


def test_compact_takes_device_or_pinned_host_rows_only(monkeypatch):
    """x and pos of up.compact may be CUDA tensors or pinned host tensors (read
    in place by the kernel); an ordinary host tensor raises before the C
    library is reached.  (The pinned case needs a GPU; see the GPU tests.)"""
    import torch

    def no_library():
        raise AssertionError("the C library was reached")

    monkeypatch.setattr(up, "lib", no_library)
    T, H, G = 128, 16, 64
    rows = torch.zeros(T, H, dtype=torch.bfloat16)
    pos = torch.zeros(T, dtype=torch.int32)
    with pytest.raises(ValueError, match="pinned host tensor"):
        up._need_rows(rows, "x", torch.bfloat16, None)
    with pytest.raises(ValueError, match="pinned host tensor"):
        up._need_rows(pos, "pos", torch.int32, None)
    with pytest.raises(TypeError, match="x must be"):
        up._need_rows(rows.float(), "x", torch.bfloat16, None)
    with pytest.raises(ValueError, match="CUDA"):  # the keep flags must be on a GPU
        up.compact(rows, pos, torch.tensor([0, T], dtype=torch.int32), G,
                   torch.zeros(2, dtype=torch.uint8), torch.tensor([0, 2], dtype=torch.int32))
