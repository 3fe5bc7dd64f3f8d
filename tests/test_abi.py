"""The C ABI library: it loads, exports every function include/fckl.h declares, sizes its
workspace as documented, and rejects bad arguments before touching a device.

CPU only: no call here reaches a kernel launch.
"""
import ctypes
import os
import re

import pytest

import chunked_kl_loss_gb300 as fckl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fckl.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fckl_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(fckl):
    names = declared_functions()
    assert "fckl_forward" in names and "fckl_backward" in names
    lib = ctypes.CDLL(fckl.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(fckl):
    lib = fckl.load()
    for st in range(7):
        assert lib.fckl_status_string(st)
    assert lib.fckl_status_string(99) == b"unknown status"


def test_kernel_names(fckl):
    names = fckl.kernel_names()
    assert names[:2] == ["preprocess", "fwd_logits_lse"]
    assert "bwd_dW_gemm" in names


def test_workspace_size_rules(fckl):
    ws = fckl.workspace_bytes
    a = ws(32768, 3072, 128256, 100, 2048, fckl.BF16)
    b = ws(65536, 3072, 128256, 100, 2048, fckl.BF16)
    c = ws(131072, 3072, 128256, 100, 2048, fckl.BF16)
    assert a > 2048 * 128256 * 2  # holds at least the bf16 gradient slab of one chunk
    # grows with N only by 4 bytes per position (per-position losses), rounded to 1 KiB
    assert abs((b - a) - 32768 * 4) <= 1024 and abs((c - b) - 65536 * 4) <= 1024
    # the chunk bounds the slab
    assert ws(32768, 3072, 128256, 100, 4096, fckl.BF16) > a
    assert ws(32768, 3072, 128256, 100, 1024, fckl.BF16) < a
    # fp32 inputs need room for their bf16 copies
    assert ws(64, 256, 4096, 16, 16, fckl.F32) > ws(64, 256, 4096, 16, 16, fckl.BF16)
    # the top-K builder's kept logits: one chunk of fp32 logits (rows padded to 256, columns to
    # a multiple of 8) and per position the list of live vocabulary tiles and its length, on top
    # of its minimum workspace (1 KiB rounding each)
    lib = fckl.load()
    for N, d, V, K, chunk in [(32768, 3072, 128256, 100, 2048), (130, 320, 2057, 100, 200)]:
        extra = (lib.fckl_topk_kept_logits_workspace_bytes(N, d, V, K, chunk, fckl.BF16)
                 - lib.fckl_topk_workspace_bytes(N, d, V, K, chunk, fckl.BF16))
        rows = -(-min(chunk, N) // 256) * 256
        tiles = -(-V // 256)
        assert 0 <= extra - rows * (-(-V // 8) * 8) * 4 - rows * tiles * 4 - rows * 4 < 3072
    # the overlap workspace: a second set of one chunk's buffers (ordered slots and their
    # masses, S and T, the three tile-statistics arrays, the gradient slab and, for fp32 inputs,
    # the chunk's bf16 H copy; 1 KiB rounding each) when there is more than one chunk
    ov = fckl.overlap_workspace_bytes
    for N, d, V, K, chunk, dt in [(32768, 3072, 128256, 100, 2048, fckl.BF16), (130, 320, 2057, 100, 100, fckl.BF16),
                                  (300, 256, 4096, 16, 64, fckl.F32)]:
        rows = -(-min(chunk, N) // 256) * 256
        tiles = -(-V // 256)
        want = 2 * rows * K * 4 + 2 * rows * 4 + 3 * tiles * rows * 4 + rows * (-(-V // 8) * 8) * 2
        regions = 8
        if dt == fckl.F32:
            want += rows * d * 2
            regions += 1
        extra = ov(N, d, V, K, chunk, dt) - ws(N, d, V, K, chunk, dt)
        assert 0 <= extra - want < regions * 1024, (extra, want)
    assert ov(2048, 256, 4096, 16, 2048, fckl.BF16) == ws(2048, 256, 4096, 16, 2048, fckl.BF16) > 0  # one chunk
    assert ov(2048, 256, 4096, 16, 4096, fckl.BF16) == ws(2048, 256, 4096, 16, 4096, fckl.BF16)
    assert ov(2049, 256, 4096, 16, 2048, fckl.BF16) > ws(2049, 256, 4096, 16, 2048, fckl.BF16)
    assert ov(0, 256, 4096, 16, 16, fckl.BF16) == 0 and ov(64, 250, 4096, 16, 16, fckl.BF16) == 0
    # the top-K builder's overlap workspace: a second set of lse, threshold, count (rows x 4 B
    # each), candidate ids and logits (rows x cmax x 4 B each), kept logits and live-tile lists
    # and their lengths, after the kept-logits workspace (1 KiB rounding each), when N > chunk
    for N, d, V, K, chunk in [(32768, 3072, 128256, 100, 2048), (130, 320, 2057, 100, 40)]:
        rows = -(-min(chunk, N) // 256) * 256
        tiles = -(-V // 256)
        cmax = V if K > tiles else min(V, 2048)
        want = 3 * rows * 4 + 2 * rows * cmax * 4 + rows * (-(-V // 8) * 8) * 4 + rows * tiles * 4 + rows * 4
        extra = (lib.fckl_topk_overlap_workspace_bytes(N, d, V, K, chunk, fckl.BF16)
                 - lib.fckl_topk_kept_logits_workspace_bytes(N, d, V, K, chunk, fckl.BF16))
        assert 0 <= extra - want < 8 * 1024, (extra, want)
    assert (lib.fckl_topk_overlap_workspace_bytes(100, 64, 1000, 8, 100, fckl.BF16)
            == lib.fckl_topk_kept_logits_workspace_bytes(100, 64, 1000, 8, 100, fckl.BF16) > 0)
    assert lib.fckl_topk_overlap_workspace_bytes(0, 64, 1000, 8, 100, fckl.BF16) == 0
    # outside the limits: 0
    assert ws(0, 256, 4096, 16, 16, fckl.BF16) == 0
    assert ws(64, 250, 4096, 16, 16, fckl.BF16) == 0  # d % 8 != 0
    assert ws(64, 256, 16, 17, 16, fckl.BF16) == 0    # K > V
    assert ws(64, 256, 4096, 1025, 16, fckl.BF16) == 0
    assert ws(64, 256, 4096, 16, 0, fckl.BF16) == 0
    assert ws(64, 256, 4096, 16, 16, 7) == 0
    # a chunk whose row count (rounded up to 256) no longer fits the int arithmetic of the
    # layout is refused, also through the no-workspace forward; min(chunk, N) is what counts
    big = (1 << 24) + 1
    assert ws(1 << 30, 256, 4096, 16, big, fckl.BF16) == 0
    assert ws(1 << 30, 256, 4096, 16, 2**31 - 1, fckl.BF16) == 0
    assert ws(4096, 256, 4096, 16, 2**31 - 1, fckl.BF16) == ws(4096, 256, 4096, 16, 4096, fckl.BF16) > 0
    assert lib.fckl_topk_workspace_bytes(1 << 30, 256, 4096, 16, big, fckl.BF16) == 0


def test_argument_errors_launch_nothing(fckl):
    lib = fckl.load()
    before = lib.fckl_launch_count()
    p = ctypes.c_void_p(256)  # never dereferenced: the checks fail first
    z = ctypes.c_void_p(0)
    # bad sizes
    assert lib.fckl_forward(p, p, 0, p, p, z, 0, 256, 4096, 16, 16, p, p, z, p, 1 << 30, z) == fckl.ERR_ARG
    assert lib.fckl_forward(p, p, 0, p, p, z, 64, 250, 4096, 16, 16, p, p, z, p, 1 << 30, z) == \
        fckl.ERR_UNSUPPORTED
    # null input
    assert lib.fckl_forward(z, p, 0, p, p, z, 64, 256, 4096, 16, 16, p, p, z, p, 1 << 30, z) == fckl.ERR_ARG
    # misaligned H
    assert lib.fckl_forward(ctypes.c_void_p(258), p, 0, p, p, z, 64, 256, 4096, 16, 16, p, p, z, p, 1 << 30,
                            z) == fckl.ERR_ARG
    # workspace too small
    assert lib.fckl_forward(p, p, 0, p, p, z, 64, 256, 4096, 16, 16, p, p, z, p, 16, z) == fckl.ERR_WORKSPACE
    assert lib.fckl_backward(p, p, 0, p, p, z, p, 64, 256, 4096, 16, 16, ctypes.c_float(1.0), p, p, p, 16,
                             z) == fckl.ERR_WORKSPACE
    assert lib.fckl_forward_backward(p, p, 0, p, p, z, 64, 256, 4096, 16, 16, ctypes.c_float(1.0), p, p, z, p,
                                     p, p, 16, z) == fckl.ERR_WORKSPACE
    # a chunk above 2^24 rows
    assert lib.fckl_forward(p, p, 0, p, p, z, 1 << 30, 256, 4096, 16, (1 << 24) + 1, p, p, z, p, 1 << 62,
                            z) == fckl.ERR_UNSUPPORTED
    assert lib.fckl_selftest_wait_timeout(p, 16, z) == fckl.ERR_ARG
    assert lib.fckl_check(z, z) == fckl.ERR_ARG
    assert lib.fckl_launch_count() == before


def test_missing_library_fails_loudly(monkeypatch):
    import importlib
    import chunked_kl_loss_gb300 as m
    monkeypatch.setattr(m, "LIB_PATH", "/nonexistent/libfckl.so")
    monkeypatch.setattr(m, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        m.load()
    importlib.reload(m)
