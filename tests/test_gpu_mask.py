"""fa_create_block_mask on the GPU vs the oracle: every table bit-exact (counts, ascending ids, zero fill,
the query-side transpose and the class matrix), on the pages' worked examples, a sweep of rules with
ragged tails and small blocks, broadcast variants, and the five workloads at full size."""
import json
import os

import numpy as np
import pytest
import torch

from block_sparse_masked_create_gb300 import fa, workloads
from oracle import flexmask_oracle as orc
from tests.gpu_common import assert_row_order, assert_tables_equal, tables_np

pytestmark = pytest.mark.gpu

CW = lambda w: [("causal",), ("window", w), ("and",)]


def gpu_tables(spec, B, H, q_len, kv_len, bq, bk, doc=None, q_off=None, bdep=None, hdep=False):
    doc_t = None if doc is None else torch.from_numpy(np.ascontiguousarray(doc, dtype=np.int32)).cuda()
    off_t = None if q_off is None else torch.from_numpy(np.ascontiguousarray(q_off, dtype=np.int32)).cuda()
    rule = fa.make_mask_rule(spec, doc_ids=doc_t, q_offset=off_t, batch_dependent=bdep, head_dependent=hdep)
    bm = fa.create_block_mask(rule, B, H, q_len, kv_len, bq, bk, keep=[doc_t, off_t])
    torch.cuda.synchronize()
    return bm, tables_np(bm)


def test_worked_example_n8_w4(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "n8_w4_2x2.json")))
    bm, t = gpu_tables(CW(4), 1, 1, 8, 8, 2, 2)
    want = orc.block_mask(CW(4), 1, 1, 8, 8, 2, 2)
    assert_tables_equal(t, want)
    h = g["hand_derived_tables"]
    assert t["kv_num"][0, 0].tolist() == h["kv_num"] and t["full_kv_num"][0, 0].tolist() == h["full_kv_num"]
    assert t["q_num"][0, 0].tolist() == h["q_num"] and t["full_q_num"][0, 0].tolist() == h["full_q_num"]
    st = fa.block_mask_stats(bm).cpu().tolist()
    assert st[:3] == [3, 6, 7]                      # full, partial, empty: 9 executed blocks, 7 empty


def test_worked_example_n16_w8(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "n16_w8_4x4.json")))
    _, t = gpu_tables(CW(8), 1, 1, 16, 16, 4, 4)
    names = {0: "empty", 1: "partial", 2: "full"}
    assert [names[int(x)] for x in t["block_class"][0, 0, -1]] == g["last_row_classes_by_kv_block"]
    assert_tables_equal(t, orc.block_mask(CW(8), 1, 1, 16, 16, 4, 4))


RULES = [
    [("causal",)], CW(5), CW(1), [("true",)], [("prefix", 0)],
    [("causal",), ("prefix", 7), ("or",)],
    [("window", 6), ("prefix", 3), ("or",)],
    [("causal",), ("doc",), ("and",)],
    [("causal",), ("prefix", 9), ("or",), ("doc",), ("and",)],
    [("doc",), ("window", 4), ("and",), ("prefix", 2), ("or",)],
]


@pytest.mark.parametrize("ri", range(len(RULES)))
@pytest.mark.parametrize("q_len,kv_len,bq,bk", [(37, 37, 8, 8), (100, 61, 16, 32), (1, 5, 4, 4), (130, 130, 128, 128),
                                                 (77, 200, 3, 7), (256, 256, 64, 128), (300, 300, 128, 16)])
def test_rule_sweep_ragged(ri, q_len, kv_len, bq, bk):
    spec = RULES[ri]
    n = max(q_len, kv_len)
    lens = np.array([5, 9, 1, 12, 7, 6, 30, 2, 50, 3, 80, 100, 100])
    doc = np.repeat(np.arange(len(lens), dtype=np.int32), lens)[:n]
    doc = np.concatenate([doc, np.full(n - len(doc), 99, np.int32)])[None, :] if len(doc) < n else doc[None, :]
    uses_doc = any(op[0] == "doc" for op in spec)
    _, t = gpu_tables(spec, 1, 1, q_len, kv_len, bq, bk, doc=doc if uses_doc else None)
    want = orc.block_mask(spec, 1, 1, q_len, kv_len, bq, bk, doc_ids=doc if uses_doc else None)
    assert_tables_equal(t, want)


@pytest.mark.parametrize("ri", [7, 8, 9])
@pytest.mark.parametrize("q_len,kv_len,bq,bk,ndoc", [(130, 130, 16, 16, 3), (256, 256, 64, 128, 40), (77, 200, 8, 4, 2)])
def test_rule_sweep_unsorted_docs(ri, q_len, kv_len, bq, bk, ndoc):
    # document ids in no particular order: row and column id ranges overlap in most blocks, so the
    # builder must visit pairs to tell partial from empty and full
    spec = RULES[ri]
    rng = np.random.default_rng(1000 * ri + q_len + ndoc)
    doc = rng.integers(0, ndoc, size=(1, max(q_len, kv_len))).astype(np.int32)
    _, t = gpu_tables(spec, 1, 1, q_len, kv_len, bq, bk, doc=doc)
    assert_tables_equal(t, orc.block_mask(spec, 1, 1, q_len, kv_len, bq, bk, doc_ids=doc))


@pytest.mark.parametrize("sorted_ids", [True, False])
def test_docs_with_rows_past_the_id_array(sorted_ids):
    # query offsets push rows past the document-id array (their id reads as -1); some key ids are -1 too
    B, H, q_len, kv_len = 2, 1, 24, 64
    off = np.array([30, 50], dtype=np.int32)
    rng = np.random.default_rng(11 + sorted_ids)
    doc = rng.integers(-1, 3, size=(B, kv_len)).astype(np.int32)
    if sorted_ids:
        doc = np.sort(doc, axis=1)
    spec = [("causal",), ("doc",), ("and",)]
    _, t = gpu_tables(spec, B, H, q_len, kv_len, 8, 8, doc=doc, q_off=off, bdep=True)
    assert_tables_equal(t, orc.block_mask(spec, B, H, q_len, kv_len, 8, 8, batch_dependent=True, q_offset=off,
                                          doc_ids=doc))


def test_batch_dependent_offsets_and_docs():
    B, H = 3, 2
    off = np.array([0, 17, 40], dtype=np.int32)
    rng = np.random.default_rng(5)
    doc = np.stack([np.sort(rng.integers(0, 4, size=64)).astype(np.int32) for _ in range(B)])
    spec = [("causal",), ("doc",), ("and",)]
    _, t = gpu_tables(spec, B, H, 20, 64, 4, 8, doc=doc, q_off=off, bdep=True)
    want = orc.block_mask(spec, B, H, 20, 64, 4, 8, batch_dependent=True, q_offset=off, doc_ids=doc)
    assert_tables_equal(t, want)
    _, th = gpu_tables([("causal",)], 1, 3, 24, 24, 8, 8, hdep=True)
    assert_tables_equal(th, orc.block_mask([("causal",)], 1, 3, 24, 24, 8, 8, head_dependent=True))


@pytest.mark.parametrize("name", ["cfg1", "cfg2", "cfg3", "cfg4b"])
def test_workload_tables(name):
    w = {"cfg1": workloads.cfg1, "cfg2": workloads.cfg2, "cfg3": workloads.cfg3,
         "cfg4b": lambda: workloads.cfg4(n=8192)}[name]()
    bm, t = gpu_tables(w.rule, w.B, w.Hq, w.q_len, w.kv_len, w.bq, w.bk, doc=w.doc_ids)
    want = orc.block_mask(w.rule, w.B, w.Hq, w.q_len, w.kv_len, w.bq, w.bk, doc_ids=w.doc_ids)
    assert_tables_equal(t, want)
    assert_row_order(t, want)
    st = fa.block_mask_stats(bm).cpu().tolist()
    cls = want["block_class"]
    assert st[0] == int((cls == 2).sum()) and st[1] == int((cls == 1).sum()) and st[2] == int((cls == 0).sum())
    if name == "cfg1":
        assert (st[0], st[1]) == (7, 14)
    if name == "cfg2":
        assert (st[0], st[1], st[2]) == (496, 32, 496)
    if name == "cfg4b":
        assert (st[0], st[1]) == (420, 120)


def test_cfg4_full_size_table():
    w = workloads.cfg4()
    bm, t = gpu_tables(w.rule, 1, w.Hq, w.q_len, w.kv_len, 128, 128)
    st = fa.block_mask_stats(bm).cpu().tolist()
    assert (st[0], st[1], st[3]) == (3556, 1016, 9)       # full, partial, longest row (window 1024 / 128 + 1)
    rows = sorted({0, 1, 7, 8, 9, 100, 255, 256, 511} | set(np.random.default_rng(4).integers(0, 512, 24).tolist()))
    want = orc.block_mask(w.rule, 1, w.Hq, w.q_len, w.kv_len, 128, 128, rows=rows)
    assert_tables_equal(t, want, rows=rows)
    # the transpose agrees with the forward table (checked on the whole table, on the device copy)
    dense_f = np.zeros((512, 512), bool)
    dense_t = np.zeros((512, 512), bool)
    for r in range(512):
        dense_f[r, t["kv_idx"][0, 0, r, :t["kv_num"][0, 0, r]]] = True
    for c in range(512):
        dense_t[t["q_idx"][0, 0, c, :t["q_num"][0, 0, c]], c] = True
    assert np.array_equal(dense_f, dense_t)


def test_cfg5_decode_table():
    d = workloads.cfg5()
    off = d.q_offset
    _, t = gpu_tables(d.rule, d.Bz, d.Hq, 1, d.kv_len, 1, d.page, q_off=off, bdep=True)
    want = orc.block_mask(d.rule, d.Bz, d.Hq, 1, d.kv_len, 1, d.page, batch_dependent=True, q_offset=off)
    assert_tables_equal(t, want)
    L = d.kv_lens
    assert np.array_equal(t["full_kv_num"][:, 0, 0], L // 128)
    assert np.array_equal(t["kv_num"][:, 0, 0], (L % 128 != 0).astype(np.int32))
    dp = workloads.cfg5(prefix=512)
    _, tp = gpu_tables(dp.rule, dp.Bz, dp.Hq, 1, dp.kv_len, 1, dp.page, q_off=off, bdep=True)
    assert_tables_equal(tp, t)      # the prefix region is already visible at every cur_pos >= 1023


def _random_rule(rng):
    """An OR of one to three AND-terms over causal / window / prefix / document atoms."""
    def atom():
        k = rng.integers(0, 4)
        if k == 0:
            return [("causal",)]
        if k == 1:
            return [("window", int(rng.integers(1, 90)))]
        if k == 2:
            return [("prefix", int(rng.integers(0, 120)))]
        return [("doc",)]

    def term():  # at most 3 ops, so a rule stays within 16 ops and 8 OR-terms
        ops = atom()
        for _ in range(int(rng.integers(0, 2))):
            ops += atom() + [("and",)]
        return ops

    spec = term()
    for _ in range(int(rng.integers(0, 3))):
        spec += term() + [("or",)]
    return spec


@pytest.mark.parametrize("seed", range(40))
def test_hull_random_rules(seed):
    # the builder skips blocks outside each row's (column's) interval hull: random OR / AND rules over
    # many blocks, per-request query offsets (which push rows past the end of the id array), sorted ids
    # with a leading -1 run, and unsorted ids on some seeds
    rng = np.random.default_rng(7000 + seed)
    spec = _random_rule(rng)
    B = 2
    q_len, kv_len = int(rng.integers(1, 500)), int(rng.integers(1, 700))
    bq, bk = int(rng.choice([1, 8, 16, 64, 128])), int(rng.choice([4, 16, 32, 128]))
    off = rng.integers(0, 300, size=B).astype(np.int32)
    n_doc = kv_len + int(rng.integers(0, 400))  # ids cover the keys; offset rows may pass the end
    doc = np.sort(rng.integers(-1, 12, size=(B, n_doc)), axis=1).astype(np.int32)
    if seed % 5 == 4:
        rng.shuffle(doc, axis=1)
    uses_doc = any(op[0] == "doc" for op in spec)
    _, t = gpu_tables(spec, B, 1, q_len, kv_len, bq, bk, doc=doc if uses_doc else None, q_off=off, bdep=True)
    want = orc.block_mask(spec, B, 1, q_len, kv_len, bq, bk, batch_dependent=True, q_offset=off,
                          doc_ids=doc if uses_doc else None)
    assert_tables_equal(t, want)
    assert_row_order(t, want)


def test_long_window_table_o_visited():
    # N = 262144, causal window 1024, 128x128 blocks: 2048 x 2048 blocks of which ~9 per row are
    # visited. Counts by closed form, sampled rows and columns against the oracle.
    N, W, bs = 262144, 1024, 128
    spec = CW(W)
    bm, t = gpu_tables(spec, 1, 1, N, N, bs, bs)
    nb = N // bs
    st = fa.block_mask_stats(bm).cpu().tolist()
    # row r >= 8: blocks r-8 (partial), r-7 .. r-1 (full), r (partial); rows 0..7 fewer
    full = sum(max(0, min(r, 7)) for r in range(nb))
    partial = sum(1 + (r >= 8) for r in range(nb))
    assert (st[0], st[1], st[3]) == (full, partial, 9)
    rows = [0, 1, 7, 8, 9, 1000, 2046, 2047]
    want = orc.block_mask(spec, 1, 1, N, N, bs, bs, rows=rows)
    assert_tables_equal(t, want, rows=rows)
    for c in (0, 5, 1000, 2040, 2047):
        # the query-side transpose of column c: rows c and c+8 partial, c+1 .. c+7 full (clipped)
        want_p = [r for r in (c, c + 8) if r < nb]
        want_f = list(range(c + 1, min(c + 8, nb)))
        assert t["q_idx"][0, 0, c, :t["q_num"][0, 0, c]].tolist() == want_p
        assert t["full_q_idx"][0, 0, c, :t["full_q_num"][0, 0, c]].tolist() == want_f
        assert not t["q_idx"][0, 0, c, len(want_p):].any() and not t["full_q_idx"][0, 0, c, len(want_f):].any()
