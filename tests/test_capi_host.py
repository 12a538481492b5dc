"""CPU-only checks of the C ABI: the library loads, exports every entry point
the header declares, and rejects bad arguments on the host before anything
would be launched (no GPU is touched: every call below fails validation)."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_117_gb300 as pkv
from paged_kv_cache_117_gb300 import build as pbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")

OK, NULL, SHAPE, DTYPE, RANGE, ALIAS, CUDA, WS, ALIGN, NO_BLOCKS = range(10)
F16, BF16, F32 = 0, 1, 2


@pytest.fixture(scope="module")
def lib():
    pbuild.build()
    return pkv.load()


def declared_functions():
    names = set()
    for fn in os.listdir(HEADER_DIR):
        if fn.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            for m in re.finditer(r"\b([a-z_][a-z0-9_]*)\s*\(", text):
                if m.group(1) not in ("sizeof", "defined"):
                    names.add(m.group(1))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert set(pkv.EXPORTED_SYMBOLS) <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared but not exported"


def test_status_strings(lib):
    for code in range(10):
        assert lib.pkv_status_string(code) != b"unknown status"
    assert lib.pkv_status_string(99) == b"unknown status"


def _expected_ws(S, Hq, D, ctx, pt):
    r = lambda x: -(-x // 256) * 256
    P = 1 if pt == 0 else max(1, -(-ctx // pt))
    n = 256 + r(4 * S * Hq) + r(8 * S * P)
    return n + (4 * S * Hq * P * (D + 2) if P > 1 else 0)


def test_workspace_bytes(lib):
    # Llama-shaped batch: 256 seqs x 32 heads x 16 partitions x (128 + 2) floats + control
    assert lib.paged_attention_workspace_bytes(256, 32, 128, 8192, 512) == \
        256 + 256 * 32 * 4 + 256 * 16 * 8 + 256 * 32 * 16 * 130 * 4
    for args in [(256, 32, 128, 8192, 0), (4, 4, 64, 512, 512), (4, 4, 64, 513, 512),
                 (3, 5, 128, 100, 16), (1, 1, 64, 16, 16)]:
        assert lib.paged_attention_workspace_bytes(*args) == _expected_ws(*args), args
    assert lib.paged_attention_workspace_bytes(-1, 4, 64, 512, 16) == ctypes.c_size_t(-1).value


P = 1 << 20            # fake, never-dereferenced, 16-byte aligned addresses
def fake(i): return P * (i + 1)


def decode(lib, **kw):
    a = dict(out=fake(0), out_dt=F32, q=fake(1), k=fake(2), v=fake(3), dt=BF16, tab=fake(4),
             max_blocks=4, lens=fake(5), S=2, Hq=8, Hkv=2, D=128, B=16, N=8, scale=0.1,
             pt=0, ws=fake(6), ws_bytes=1 << 20)
    a.update(kw)
    return lib.paged_attention_decode(a["out"], a["out_dt"], a["q"], a["k"], a["v"], a["dt"],
                                      a["tab"], a["max_blocks"], a["lens"], a["S"], a["Hq"],
                                      a["Hkv"], a["D"], a["B"], a["N"], a["scale"], a["pt"],
                                      a["ws"], a["ws_bytes"], None)


def test_decode_validation(lib):
    assert decode(lib, q=None) == NULL
    assert decode(lib, dt=F32) == DTYPE
    assert decode(lib, out_dt=7) == DTYPE
    assert decode(lib, D=96) == SHAPE
    assert decode(lib, B=12) == SHAPE
    assert decode(lib, Hq=6, Hkv=4) == SHAPE
    assert decode(lib, pt=24) == SHAPE
    assert decode(lib, S=-1) == RANGE
    assert decode(lib, S=70000) == RANGE
    assert decode(lib, q=fake(1) + 8) == ALIGN
    assert decode(lib, k=fake(2), v=fake(2)) == ALIAS
    assert decode(lib, out=fake(1)) == ALIAS
    assert decode(lib, ws=None) == WS
    assert decode(lib, ws_bytes=10) == WS
    assert decode(lib, ws=fake(6) + 16) == ALIGN
    assert decode(lib, ws=fake(1)) == ALIAS
    assert decode(lib, S=0) == OK           # nothing to do: returns before any CUDA call


def append(lib, **kw):
    a = dict(out=fake(0), out_dt=F32, q=fake(1), key=fake(7), val=fake(8), k=fake(2), v=fake(3),
             dt=BF16, tab=fake(4), max_blocks=4, lens=fake(5), S=2, Hq=8, Hkv=2, D=128, B=16,
             N=8, scale=0.1, pt=0, ws=fake(6), ws_bytes=1 << 20)
    a.update(kw)
    return lib.paged_attention_decode_append(
        a["out"], a["out_dt"], a["q"], a["key"], a["val"], a["k"], a["v"], a["dt"], a["tab"],
        a["max_blocks"], a["lens"], a["S"], a["Hq"], a["Hkv"], a["D"], a["B"], a["N"],
        a["scale"], a["pt"], a["ws"], a["ws_bytes"], None)


def test_decode_append_validation(lib):
    assert append(lib, key=None) == NULL
    assert append(lib, val=None) == NULL
    assert append(lib, q=None) == NULL
    assert append(lib, key=fake(7) + 8) == ALIGN
    assert append(lib, key=fake(2) + 256) == ALIAS          # inside the K pool
    assert append(lib, val=fake(3)) == ALIAS                # the V pool itself
    assert append(lib, key=fake(0) + 64) == ALIAS           # the output
    assert append(lib, val=fake(6) + 512) == ALIAS          # the workspace
    assert append(lib, D=96) == SHAPE
    assert append(lib, ws=None) == WS
    assert append(lib, S=0) == OK
    assert append(lib, S=0, key=None, val=None) == OK       # nothing to append or read


def chunked(lib, **kw):
    a = dict(out=fake(0), out_dt=F32, q=fake(1), k=fake(2), v=fake(3), dt=BF16, tab=fake(4),
             max_blocks=4, lens=fake(5), qs=fake(6), S=2, T=64, maxq=32, Hq=8, Hkv=2, D=128,
             B=16, N=8, scale=0.1, pf=0)
    a.update(kw)
    return lib.paged_attention_chunked(a["out"], a["out_dt"], a["q"], a["k"], a["v"], a["dt"],
                                       a["tab"], a["max_blocks"], a["lens"], a["qs"], a["S"],
                                       a["T"], a["maxq"], a["Hq"], a["Hkv"], a["D"], a["B"],
                                       a["N"], a["scale"], a["pf"], None)


def test_chunked_validation(lib):
    assert chunked(lib, q=None) == NULL
    assert chunked(lib, qs=None) == NULL
    assert chunked(lib, dt=F32) == DTYPE
    assert chunked(lib, out_dt=7) == DTYPE
    assert chunked(lib, pf=2) == DTYPE
    assert chunked(lib, D=96) == SHAPE
    assert chunked(lib, B=12) == SHAPE
    assert chunked(lib, B=4) == SHAPE
    assert chunked(lib, Hq=6, Hkv=4) == SHAPE
    assert chunked(lib, Hq=256, Hkv=1) == SHAPE          # group above 128
    assert chunked(lib, S=-1) == RANGE
    assert chunked(lib, maxq=65) == RANGE                 # more rows than the batch holds
    assert chunked(lib, q=fake(1) + 8) == ALIGN
    assert chunked(lib, out=fake(0) + 8) == ALIGN         # rows are stored 16 bytes at a time
    assert chunked(lib, qs=fake(6) + 2) == ALIGN
    assert chunked(lib, k=fake(2), v=fake(2)) == ALIAS
    assert chunked(lib, out=fake(1)) == ALIAS
    assert chunked(lib, out=fake(6)) == ALIAS             # output over query_start
    assert chunked(lib, T=0, maxq=0) == OK                # nothing to do: no CUDA call
    assert chunked(lib, S=0) == OK


def mixed(lib, **kw):
    a = dict(out=fake(0), out_dt=F32, q=fake(1), k=fake(2), v=fake(3), dt=BF16, tab=fake(4),
             max_blocks=4, lens=fake(5), qs=fake(6), S=2, T=64, maxq=32, Hq=8, Hkv=2, D=128,
             B=16, N=8, scale=0.1, pf=0, pt=32, ws=fake(7), ws_bytes=1 << 20)
    a.update(kw)
    return lib.paged_attention_mixed(a["out"], a["out_dt"], a["q"], a["k"], a["v"], a["dt"],
                                     a["tab"], a["max_blocks"], a["lens"], a["qs"], a["S"],
                                     a["T"], a["maxq"], a["Hq"], a["Hkv"], a["D"], a["B"],
                                     a["N"], a["scale"], a["pf"], a["pt"], a["ws"],
                                     a["ws_bytes"], None)


def test_mixed_validation(lib):
    """paged_attention_mixed checks the chunked half's arguments and the decode
    half's (partition, workspace) before anything is launched."""
    assert mixed(lib, q=None) == NULL
    assert mixed(lib, qs=None) == NULL
    assert mixed(lib, pf=2) == DTYPE
    assert mixed(lib, B=4) == SHAPE                       # the chunked half needs blocks of 8+
    assert mixed(lib, pt=24) == SHAPE                     # partition not a multiple of the block
    assert mixed(lib, maxq=65) == RANGE
    assert mixed(lib, ws=None) == WS
    assert mixed(lib, ws_bytes=64) == WS
    assert mixed(lib, ws=fake(7) + 16) == ALIGN
    assert mixed(lib, ws=fake(0)) == ALIAS                # the workspace over the output
    assert mixed(lib, out=fake(6)) == ALIAS               # the output over query_start
    assert mixed(lib, T=0, maxq=0) == OK                  # nothing to do: no CUDA call
    assert mixed(lib, S=0) == OK


def test_write_validation(lib):
    f = lib.paged_kv_write
    assert f(None, fake(1), fake(2), fake(3), fake(4), 4, 8, 16, 2, 128, BF16, None) == NULL
    assert f(fake(0), fake(1), fake(2), fake(3), fake(4), 4, 8, 16, 2, 128, F32, None) == DTYPE
    assert f(fake(0), fake(1), fake(2), fake(3), fake(4), 4, 8, 16, 2, 100, BF16, None) == SHAPE
    assert f(fake(0), fake(1), fake(2), fake(3), fake(4), -1, 8, 16, 2, 128, BF16, None) == RANGE
    assert f(fake(0) + 4, fake(1), fake(2), fake(3), fake(4), 4, 8, 16, 2, 128, BF16, None) == ALIGN
    assert f(fake(0), fake(1), fake(2), fake(2), fake(4), 4, 8, 16, 2, 128, BF16, None) == ALIAS
    assert f(fake(0), fake(1), fake(2), fake(3), fake(4), 0, 8, 16, 2, 128, BF16, None) == OK


def test_copy_validation(lib):
    f = lib.paged_block_copy
    assert f(None, fake(1), fake(2), 3, 8, 16, 2, 128, BF16, None) == NULL
    assert f(fake(0), fake(1), fake(2), 3, 8, 16, 2, 128, 5, None) == DTYPE
    assert f(fake(0), fake(1), fake(2), 3, 8, 20, 2, 128, BF16, None) == SHAPE
    assert f(fake(0), fake(1), fake(2), -3, 8, 16, 2, 128, BF16, None) == RANGE
    assert f(fake(0), fake(1), fake(2) + 4, 3, 8, 16, 2, 128, BF16, None) == ALIGN
    assert f(fake(0), fake(0), fake(2), 3, 8, 16, 2, 128, BF16, None) == ALIAS
    assert f(fake(0), fake(1), fake(2), 0, 8, 16, 2, 128, BF16, None) == OK


def test_copy_ws_validation(lib):
    """paged_block_copy_ws: the counter workspace is checked on the host (present,
    large enough, aligned, apart from the pools and the pairs) before any launch."""
    f = lib.paged_block_copy_ws
    assert lib.paged_block_copy_workspace_bytes(8) == 256
    assert lib.paged_block_copy_workspace_bytes(40_000) == 320_000
    assert lib.paged_block_copy_workspace_bytes(0) == ctypes.c_size_t(-1).value
    ws = fake(5)
    args = lambda **kw: [kw.get("k", fake(0)), fake(1), fake(2), kw.get("P", 3), 8, 16, 2, 128,
                         BF16, kw.get("ws", ws), kw.get("n", 256), None]
    assert f(*args(ws=None)) == WS
    assert f(*args(n=255)) == WS
    assert f(*args(ws=ws + 16)) == ALIGN
    assert f(*args(ws=fake(0) + 256)) == ALIAS       # inside the K pool
    assert f(*args(k=None)) == NULL
    assert f(*args(P=0)) == OK                        # nothing to copy: no launch


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="CUDA library not found"):
        pkv.load(str(tmp_path / "missing.so"))
