"""The C-ABI library: it builds, loads without a GPU, exports every symbol include/fa.h declares, and its
host-side checks reject bad arguments before launching anything (no GPU needed for any of this)."""
import ctypes
import os
import re

import pytest

from block_sparse_masked_create_gb300 import build as fa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    from block_sparse_masked_create_gb300 import fa
    return fa.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "fa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:FA_API\s+)?(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s+\**(fa_[a-z0-9_]+)\s*\(",
                       src, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"fa_create_block_mask", "fa_flex_forward", "fa_flex_decode"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"


def test_version_and_status_strings(lib):
    from block_sparse_masked_create_gb300 import fa
    assert b"sm_103a" in lib.fa_version()
    assert fa.status_string(fa.ERR_TIMEOUT) == "device wait timed out"


def test_host_side_rejections_launch_nothing(lib):
    from block_sparse_masked_create_gb300 import fa
    r = fa.make_mask_rule([("causal",)])
    # sizes: table bytes are a pure host computation
    n = fa.block_mask_bytes(r, 4, 16, 4096, 4096, 128, 128)
    assert n >= 4 * 32 * 32 * 4 + 32 * 32
    assert fa.block_mask_bytes(r, 1, 1, 0, 8, 2, 2) == 0            # Q_LEN < 1
    assert fa.block_mask_bytes(r, 1, 1, 8, 8, 129, 2) == 0          # Bq > 128
    c = fa.BlockMaskC()
    dummy = ctypes.c_void_p(256)                                    # never dereferenced: rejected first
    bad = fa.make_mask_rule([("causal",), ("and",)])                # malformed postfix program
    assert lib.fa_create_block_mask(ctypes.byref(bad), 1, 1, 8, 8, 2, 2, dummy, 1 << 20, ctypes.byref(c), None) \
        == fa.ERR_INVALID_ARG
    assert lib.fa_create_block_mask(ctypes.byref(r), 1, 1, 8, 8, 2, 2, dummy, 16, ctypes.byref(c), None) \
        == fa.ERR_BUFFER
    doc_rule = fa.make_mask_rule([("causal",), ("doc",), ("and",)])  # doc op without doc ids
    assert lib.fa_create_block_mask(ctypes.byref(doc_rule), 1, 1, 8, 8, 2, 2, dummy, 1 << 20, ctypes.byref(c),
                                    None) == fa.ERR_INVALID_ARG
    many = fa.make_mask_rule([("causal",), ("doc",), ("or",)] +
                             [op for w in (1, 2, 3) for op in (("window", w), ("prefix", w), ("or",), ("and",))])
    # (causal | doc) & (w1 | p1) & (w2 | p2) & (w3 | p3): more than 8 distinct conjunctions
    assert lib.fa_create_block_mask(ctypes.byref(many), 1, 1, 8, 8, 2, 2, dummy, 1 << 20, ctypes.byref(c), None) \
        == fa.ERR_UNSUPPORTED


def test_forward_and_decode_argument_checks(lib):
    from block_sparse_masked_create_gb300 import fa
    c = fa.BlockMaskC()
    c.Bm, c.Hm, c.q_len, c.kv_len, c.bq, c.bk, c.nq, c.nk = 1, 1, 256, 256, 128, 128, 2, 2
    for name in ("kv_num", "kv_idx", "full_kv_num", "full_kv_idx"):
        setattr(c, name, 4096)
    c.rule = fa.make_mask_rule([("causal",)])
    p = ctypes.c_void_p(4096)
    f = lib.fa_flex_forward
    # length mismatch with the mask is an error, never a silent trim
    assert f(p, p, p, ctypes.byref(c), None, 0.0, p, 0, p, 1, 2, 1, 255, 256, 128, None, None, None) == fa.ERR_SHAPE
    assert f(p, p, p, ctypes.byref(c), None, 0.0, p, 0, p, 1, 3, 2, 256, 256, 128, None, None, None) == fa.ERR_SHAPE
    assert f(p, p, p, ctypes.byref(c), None, 0.0, p, 0, p, 1, 2, 1, 256, 256, 96, None, None, None) == \
        fa.ERR_UNSUPPORTED
    assert f(ctypes.c_void_p(4097), p, p, ctypes.byref(c), None, 0.0, p, 0, p, 1, 2, 1, 256, 256, 128, None, None,
             None) == fa.ERR_INVALID_ARG                             # misaligned q
    assert f(p, p, p, ctypes.byref(c), None, 0.0, p, 7, p, 1, 2, 1, 256, 256, 128, None, None, None) == \
        fa.ERR_INVALID_ARG                                           # unknown output type
    assert lib.fa_decode_workspace_bytes(64, 32, 128, 256, 128) > 64 * 32 * 128 * 4
    d = lib.fa_flex_decode
    # table made for prefill (bq = 128) is rejected by decode
    assert d(p, p, p, p, 10, ctypes.byref(c), None, 0.0, p, 0, p, 1, 4, 2, 128, 128, 2, p, 1 << 30, None, None,
             None) == fa.ERR_SHAPE


def _mask_struct(fa, nq=2, nk=2, bq=128, bk=128, q_len=256, kv_len=256):
    c = fa.BlockMaskC()
    c.Bm, c.Hm, c.q_len, c.kv_len, c.bq, c.bk, c.nq, c.nk = 1, 1, q_len, kv_len, bq, bk, nq, nk
    for name in ("kv_num", "kv_idx", "full_kv_num", "full_kv_idx", "q_num", "q_idx", "full_q_num", "full_q_idx",
                 "block_class"):
        setattr(c, name, 4096)
    c.rule = fa.make_mask_rule([("causal",)])
    return c


def test_paged_forward_argument_checks(lib):
    from block_sparse_masked_create_gb300 import fa
    c = _mask_struct(fa)
    p = ctypes.c_void_p(4096)
    f = lib.fa_flex_forward_paged
    args = lambda pt, n_pages, page, max_pages: (p, p, p, pt, n_pages, page, max_pages, ctypes.byref(c), None, 0.0,
                                                 p, 1, p, 1, 2, 1, 256, 256, 128, None, None)
    assert f(*args(None, 8, 128, 2)) == fa.ERR_INVALID_ARG               # no page table
    assert f(*args(p, 8, 64, 2)) == fa.ERR_SHAPE                         # page != Bk
    assert f(*args(p, 8, 128, 1)) == fa.ERR_SHAPE                        # table shorter than the key blocks
    assert f(*args(p, 0, 128, 2)) == fa.ERR_SHAPE                        # empty pool
    assert f(*args(ctypes.c_void_p(4098), 8, 128, 2)) == fa.ERR_INVALID_ARG  # misaligned table


def test_select_rows_argument_checks(lib):
    from block_sparse_masked_create_gb300 import fa
    c = _mask_struct(fa, nq=256, nk=256, bq=128, bk=128, q_len=32768, kv_len=32768)
    n = lib.fa_block_mask_select_bytes(ctypes.byref(c), 64)
    assert n >= 64 * 256 * 4 * 4                                         # lists, classes, one-row transpose
    c.Bm = 4
    assert lib.fa_block_mask_select_bytes(ctypes.byref(c), 64) == 0      # per-batch table of another batch
    c.Bm = 1
    out = fa.BlockMaskC()
    p = ctypes.c_void_p(4096)
    buf = ctypes.c_void_p(1 << 20)
    assert lib.fa_block_mask_select_rows(ctypes.byref(c), p, 64, buf, 16, ctypes.byref(out), None, None) == \
        fa.ERR_BUFFER
    c.rule.q_offset = 4096                                               # the prebuilt table must be global
    assert lib.fa_block_mask_select_rows(ctypes.byref(c), p, 64, buf, 1 << 30, ctypes.byref(out), None, None) == \
        fa.ERR_INVALID_ARG


def test_host_forward_argument_checks(lib):
    from block_sparse_masked_create_gb300 import fa
    ws = lib.fa_forward_host_workspace_bytes
    n = ws(4, 16, 16, 4096, 4096, 128, 1)
    assert n >= 2 * (4096 * 128 * 2 * 3 + 4096 * 128 * 4)               # at least one head's slot, twice
    assert ws(4, 16, 16, 4096, 4096, 96, 1) == 0                          # head dim
    assert ws(4, 16, 5, 4096, 4096, 128, 1) == 0                          # Hq % Hkv
    c = _mask_struct(fa)
    p = ctypes.c_void_p(4096)
    f = lib.fa_flex_forward_host
    wsn = ws(1, 2, 1, 256, 256, 128, 1)
    assert f(None, p, p, ctypes.byref(c), None, 0.0, p, 1, p, 1, 2, 1, 256, 256, 128, ctypes.c_void_p(1 << 20),
             wsn, None, None) == fa.ERR_INVALID_ARG
    assert f(p, p, p, ctypes.byref(c), None, 0.0, p, 1, p, 1, 2, 1, 256, 256, 128, ctypes.c_void_p(1 << 20),
             wsn - 1, None, None) == fa.ERR_BUFFER
    assert f(p, p, p, ctypes.byref(c), None, 0.0, p, 1, p, 1, 2, 1, 255, 256, 128, ctypes.c_void_p(1 << 20),
             1 << 30, None, None) == fa.ERR_SHAPE                         # length differs from the mask


def test_backward_argument_checks(lib):
    from block_sparse_masked_create_gb300 import fa
    c = _mask_struct(fa)
    p = ctypes.c_void_p(4096)
    f = lib.fa_flex_backward
    ok_args = lambda **kw: [kw.get("q", p), p, p, p, 1, p, p, ctypes.byref(c), None, 0.0, p, p, p, p, 1, 2, 1,
                            256, 256, kw.get("d", 128), None, None]
    assert f(*ok_args(q=None)) == fa.ERR_INVALID_ARG
    assert f(*ok_args(d=96)) == fa.ERR_UNSUPPORTED
    c.q_num = None                                                       # the transpose is required
    assert f(*ok_args()) == fa.ERR_INVALID_ARG
