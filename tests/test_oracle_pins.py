"""Pins of the fp64 oracle to what the pages and the mathematics fix (no GPU).

Each test checks the oracle against something other than itself: numbers the pages print (tests/golden/),
closed forms, library routines (torch fp64 softmax / SDPA math path on CPU) or brute-force invariants.
The mutation tests at the end plant plausible mistakes in the oracle and check that a pin catches them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import flexmask_oracle as orc

CAUSAL_WIN = lambda w: [("causal",), ("window", w), ("and",)]


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# ------------------------------------------------------------------ worked examples printed on the pages
def test_n8_w4_2x2_worked_example(golden_dir):
    g = _load(golden_dir, "n8_w4_2x2.json")
    N, W, bq, bk = g["N"], g["W"], g["bq"], g["bk"]
    rule = CAUSAL_WIN(W)
    a = orc.dense_allowed(rule, 0, np.arange(N), N, N)
    assert int(a.sum()) == g["valid_edges"]
    t = orc.block_mask(rule, 1, 1, N, N, bq, bk)
    cls = t["block_class"][0, 0]
    executed = int((cls != orc.EMPTY).sum())
    assert executed == g["executed_blocks"]
    assert executed * bq * bk == g["elements_covered_by_executed_blocks"]
    assert int((cls == orc.EMPTY).sum()) == g["empty_blocks"]
    blk = a[4:6, 0:2]
    assert [tuple(x) for x in np.argwhere(blk) + [4, 0]] == [tuple(g["block_q4_5_k0_1_only_allowed_pair"])]
    assert cls[2, 0] == orc.PARTIAL
    assert cls[2, 1] == orc.FULL and g["block_q4_5_k2_3_class"] == "full"
    h = g["hand_derived_tables"]
    for key in ("kv", "full_kv"):
        assert t[key + "_num"][0, 0].tolist() == h[key + "_num"]
        for r, lst in enumerate(h[key + "_idx"]):
            row = t[key + "_idx"][0, 0, r]
            assert row[:len(lst)].tolist() == lst and not row[len(lst):].any()
    for key in ("q", "full_q"):
        assert t[key + "_num"][0, 0].tolist() == h[key + "_num"]
        for c, lst in enumerate(h[key + "_idx"]):
            col = t[key + "_idx"][0, 0, c]
            assert col[:len(lst)].tolist() == lst and not col[len(lst):].any()


def test_n16_w8_4x4_last_row(golden_dir):
    g = _load(golden_dir, "n16_w8_4x4.json")
    t = orc.block_mask(CAUSAL_WIN(g["W"]), 1, 1, g["N"], g["N"], g["bq"], g["bk"])
    names = {orc.EMPTY: "empty", orc.PARTIAL: "partial", orc.FULL: "full"}
    last = t["block_class"][0, 0, -1]
    assert [names[int(c)] for c in last] == g["last_row_classes_by_kv_block"]
    # the same page's pair-count formula at this size: 8*9/2 + 8*8 = 100
    assert int(orc.dense_allowed(CAUSAL_WIN(8), 0, np.arange(16), 16, 16).sum()) == 100


def _count_pairs(rule, n, chunk=512):
    tot = 0
    for r0 in range(0, n, chunk):
        tot += int(orc.dense_allowed(rule, 0, np.arange(r0, min(n, r0 + chunk)), n, n).sum())
    return tot


def test_window_pair_count_closed_form(golden_dir):
    g = _load(golden_dir, "window_pairs.json")
    N, W = g["N"], g["W"]
    closed = W * (W + 1) // 2 + (N - W) * W        # the page's closed form, written out here
    assert closed == 7_864_832
    assert _count_pairs(CAUSAL_WIN(W), N) == closed
    assert _count_pairs([("causal",)], N) == N * (N + 1) // 2 == 33_558_528
    assert _count_pairs([("true",)], 2048) == 2048 * 2048 and N * N == 67_108_864
    rnd = g["printed_rounding"]
    assert abs(closed - g["printed_window_pairs_approx"]) <= rnd
    assert abs(N * N - g["printed_dense_pairs_approx"]) <= rnd
    assert abs(N * (N + 1) // 2 - g["printed_causal_pairs_approx"]) <= rnd
    # the page's small example: W=4, query 6 sees exactly 3..6
    assert np.nonzero(orc.dense_allowed(CAUSAL_WIN(4), 0, np.array([6]), 8, 8)[0])[0].tolist() == [3, 4, 5, 6]


def _closed_causal(r, c, br, bc):
    # article on causal geometric pruning, section 1: empty iff (i+1)Br-1 < jBc; full iff iBr >= (j+1)Bc-1
    if (r + 1) * br - 1 < c * bc:
        return orc.EMPTY
    if r * br >= (c + 1) * bc - 1:
        return orc.FULL
    return orc.PARTIAL


@pytest.mark.parametrize("n,br,bc", [(4096, 128, 128), (512, 64, 128), (512, 128, 64), (256, 32, 32)])
def test_causal_block_geometry(n, br, bc):
    t = orc.block_mask([("causal",)], 1, 1, n, n, br, bc)
    cls = t["block_class"][0, 0]
    want = np.array([[_closed_causal(r, c, br, bc) for c in range(n // bc)] for r in range(n // br)])
    assert np.array_equal(cls, want)
    if br == bc:
        nb = n // br
        assert int((cls == orc.PARTIAL).sum()) == nb               # min(N/Br, N/Bc) boundary blocks
        assert int((cls == orc.EMPTY).sum()) == nb * (nb - 1) // 2
    if (n, br) == (4096, 128):
        assert (int((cls == orc.FULL).sum()), int((cls == orc.PARTIAL).sum()),
                int((cls == orc.EMPTY).sum())) == (496, 32, 496)


def test_causal_geometry_figure(golden_dir):
    g = _load(golden_dir, "causal_geometry.json")
    names = {orc.EMPTY: "empty", orc.PARTIAL: "boundary", orc.FULL: "full"}
    cls = orc.block_mask([("causal",)], 1, 1, 16, 16, 4, 4)["block_class"][0, 0]
    assert [[names[int(x)] for x in row] for row in cls] == g["figure_4x4"]


def test_interval_rule_example():
    # PaperTrace 5.1.2, section 6.3: rows a=4..b=7, W=4: union [1,7], intersection {4}; KV block [2,3] partial
    a = orc.dense_allowed(CAUSAL_WIN(4), 0, np.arange(4, 8), 8, 8)
    union = np.nonzero(a.any(axis=0))[0]
    inter = np.nonzero(a.all(axis=0))[0]
    assert union.tolist() == list(range(1, 8)) and inter.tolist() == [4]
    blk = a[:, 2:4]
    assert blk.any() and not blk.all()


# ------------------------------------------------------------------ block table invariants (brute force)
RULES = [
    [("causal",)],
    CAUSAL_WIN(5),
    [("causal",), ("doc",), ("and",)],
    [("causal",), ("prefix", 7), ("or",)],
    [("causal",), ("prefix", 7), ("or",), ("doc",), ("and",)],
    [("window", 6), ("prefix", 3), ("or",)],
    [("true",)],
    [("prefix", 0)],
]


@pytest.mark.parametrize("rule", RULES)
@pytest.mark.parametrize("n,bq,bk", [(37, 8, 8), (40, 8, 4), (33, 16, 8), (1, 4, 4), (3, 2, 2)])
def test_tables_expand_to_mask(rule, n, bq, bk):
    doc = np.repeat(np.arange(6, dtype=np.int32), [5, 9, 1, 12, 7, 6])[:n][None, :] if n > 1 else \
        np.zeros((1, n), np.int32)
    if doc.shape[1] < n:
        doc = np.concatenate([doc, np.full((1, n - doc.shape[1]), 99, np.int32)], axis=1)
    t = orc.block_mask(rule, 1, 1, n, n, bq, bk, doc_ids=doc)
    nq, nk = t["nq"], t["nk"]
    a = orc.dense_allowed(rule, 0, np.arange(nq * bq), n, n, 0, doc, np.arange(nk * bk))
    m_hat = orc.expand_tables(t)[0, 0]
    assert np.all(a[m_hat == orc.FULL])                  # full blocks are all-true
    assert not np.any(a[m_hat == orc.EMPTY])             # dropped blocks are all-false
    for r in range(nq):                                  # partial blocks are mixed
        for c in range(nk):
            blk = a[r * bq:(r + 1) * bq, c * bk:(c + 1) * bk]
            if t["block_class"][0, 0, r, c] == orc.PARTIAL:
                assert blk.any() and not blk.all()
    # lists are ascending, unique, zero-filled; the transpose is the forward table transposed
    for key, numk in (("kv_idx", "kv_num"), ("full_kv_idx", "full_kv_num")):
        for r in range(nq):
            k = t[numk][0, 0, r]
            row = t[key][0, 0, r]
            assert np.all(np.diff(row[:k]) > 0) and not row[k:].any()
    for fwd, tr in (("kv", "q"), ("full_kv", "full_q")):
        dense_f = np.zeros((nq, nk), bool)
        dense_t = np.zeros((nq, nk), bool)
        for r in range(nq):
            dense_f[r, t[fwd + "_idx"][0, 0, r, :t[fwd + "_num"][0, 0, r]]] = True
        for c in range(nk):
            dense_t[t[tr + "_idx"][0, 0, c, :t[tr + "_num"][0, 0, c]], c] = True
        assert np.array_equal(dense_f, dense_t)
    if n % bq or n % bk:                                 # tail blocks are never full
        if n % bq:
            assert not np.any(t["block_class"][0, 0, -1] == orc.FULL)
        if n % bk:
            assert not np.any(t["block_class"][0, 0, :, -1] == orc.FULL)


def test_broadcast_dims():
    off = np.array([3, 9], dtype=np.int32)
    t = orc.block_mask([("causal",)], 2, 3, 4, 16, 2, 4, batch_dependent=True, q_offset=off)
    assert t["block_class"].shape == (2, 1, 2, 4)
    # request 1 (offset 9) sees positions <= 9..12 -> blocks 0,1 full, block 2 partial (8..11 vs rows 9,10)
    assert t["block_class"][1, 0, 0].tolist() == [2, 2, 1, 0]
    th = orc.block_mask([("causal",)], 1, 3, 8, 8, 4, 4, head_dependent=True)
    assert th["block_class"].shape == (1, 3, 2, 2) and np.all(th["block_class"] == th["block_class"][:, :1])


# ------------------------------------------------------------------ attention: library special cases
def _torch_dense(q, k, v, scale, causal):
    tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    s = (tq @ tk.transpose(-1, -2)) * scale
    if causal:
        n = s.shape[-1]
        s = s.masked_fill(torch.ones(n, n, dtype=torch.bool).triu(1), float("-inf"))
    return o.numpy(), torch.logsumexp(s, dim=-1).numpy()


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_fp64(causal):
    B, H, N, d = 2, 3, 45, 16
    q, k, v = _rand((B, H, N, d), 1), _rand((B, H, N, d), 2), _rand((B, H, N, d), 3)
    scale = 0.3
    o, lse = orc.attention(q, k, v, [("causal",)] if causal else [("true",)], scale=scale)
    o_ref, lse_ref = _torch_dense(q, k, v, scale, causal)
    assert np.max(np.abs(o - o_ref)) < 1e-12
    assert np.max(np.abs(lse - lse_ref)) < 1e-12


def test_default_scale_is_inverse_sqrt_d():
    q, k, v = _rand((1, 1, 9, 16), 4), _rand((1, 1, 9, 16), 5), _rand((1, 1, 9, 16), 6)
    o, _ = orc.attention(q, k, v, [("true",)])
    o_ref, _ = _torch_dense(q, k, v, 0.25, False)
    assert np.max(np.abs(o - o_ref)) < 1e-12


def test_row_sums_and_lse():
    q, k, v = _rand((12, 8), 7), _rand((30, 8), 8), _rand((30, 8), 9)
    rows = np.arange(12) + 5
    o, lse, p = orc.attention_rows(q, k, v, CAUSAL_WIN(9), rows, 0, 0, 40, 30, 0.5, return_p=True)
    assert np.all(np.abs(p.sum(axis=1) - 1.0) < 1e-12)
    a = orc.dense_allowed(CAUSAL_WIN(9), 0, rows, 40, 30)
    assert np.all(p[~a] == 0.0)
    s = 0.5 * q @ k.T
    for r in range(12):
        sr = s[r][a[r]]
        assert abs(lse[r] - (sr.max() + math.log(np.exp(sr - sr.max()).sum()))) < 1e-12


def test_gqa_equals_expanded_kv():
    B, Hq, Hkv, N, d = 1, 6, 2, 21, 8
    q, k, v = _rand((B, Hq, N, d), 10), _rand((B, Hkv, N, d), 11), _rand((B, Hkv, N, d), 12)
    slopes = np.linspace(0.1, 0.6, Hq)
    score = dict(alibi_slopes=slopes, softcap=3.0)
    o, lse = orc.attention(q, k, v, CAUSAL_WIN(7), score=score)
    ke = np.repeat(k, Hq // Hkv, axis=1)        # query head h reads KV head floor(h/g)
    ve = np.repeat(v, Hq // Hkv, axis=1)
    o2, lse2 = orc.attention(q, ke, ve, CAUSAL_WIN(7), score=score)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
    # the score rule reads the QUERY head: sibling query heads with different slopes differ
    assert not np.allclose(lse[0, 0], lse[0, 1])


def test_doc_causal_is_per_document_causal():
    lens = [5, 11, 3, 9]
    doc = np.repeat(np.arange(4, dtype=np.int32), lens)[None, :]
    N = sum(lens)
    q, k, v = _rand((1, 2, N, 8), 13), _rand((1, 2, N, 8), 14), _rand((1, 2, N, 8), 15)
    o, lse = orc.attention(q, k, v, [("causal",), ("doc",), ("and",)], scale=0.4, doc_ids=doc)
    s0 = 0
    for L in lens:
        sl = slice(s0, s0 + L)
        o_ref, lse_ref = _torch_dense(q[:, :, sl], k[:, :, sl], v[:, :, sl], 0.4, True)
        assert np.max(np.abs(o[:, :, sl] - o_ref)) < 1e-12
        assert np.max(np.abs(lse[:, :, sl] - lse_ref)) < 1e-12
        s0 += L


def test_prefix_lm():
    N, P = 24, 7
    q, k, v = _rand((1, 1, N, 8), 16), _rand((1, 1, N, 8), 17), _rand((1, 1, N, 8), 18)
    o, lse = orc.attention(q, k, v, [("causal",), ("prefix", P), ("or",)], scale=0.5)
    o_pre, lse_pre = _torch_dense(q[:, :, :P], k[:, :, :P], v[:, :, :P], 0.5, False)   # prefix: bidirectional
    assert np.max(np.abs(o[:, :, :P] - o_pre)) < 1e-12
    o_c, lse_c = _torch_dense(q, k, v, 0.5, True)                                       # later rows: causal
    assert np.max(np.abs(o[:, :, P:] - o_c[:, :, P:])) < 1e-12


# ------------------------------------------------------------------ closed forms for the score rules
def test_single_key_rows():
    # window 1: each row sees only itself -> O_i = v_i exactly, LSE_i = (scored) s_ii
    N, d = 10, 8
    q, k, v = _rand((1, 2, N, d), 19), _rand((1, 2, N, d), 20), _rand((1, 2, N, d), 21)
    c = 2.5
    o, lse = orc.attention(q, k, v, CAUSAL_WIN(1), scale=0.7, score=dict(softcap=c))
    assert np.array_equal(o, v)
    s = 0.7 * np.einsum("bhnd,bhnd->bhn", q, k)
    assert np.max(np.abs(lse - c * np.tanh(s / c))) < 1e-14
    assert np.all(np.abs(lse) < c)


def test_alibi_closed_form():
    # q = 0 -> every score is the bias -slope*(i-j); causal rows are geometric distributions
    N, H = 17, 4
    q = np.zeros((1, H, N, 4))
    k = _rand((1, H, N, 4), 22)
    v = np.broadcast_to(np.eye(N)[None, None], (1, H, N, N)).copy()      # one-hot: O row = P row
    slopes = 2.0 ** (-8.0 * (np.arange(H) + 1) / H)
    o, lse = orc.attention(q, k, v, [("causal",)], score=dict(alibi_slopes=slopes))
    for h in range(H):
        a = slopes[h]
        for i in range(N):
            want_lse = math.log((1 - math.exp(-a * (i + 1))) / (1 - math.exp(-a)))
            assert abs(lse[0, h, i] - want_lse) < 1e-12
            j = np.arange(i + 1)
            want_p = np.exp(-a * (i - j)) * (1 - math.exp(-a)) / (1 - math.exp(-a * (i + 1)))
            assert np.max(np.abs(o[0, h, i, :i + 1] - want_p)) < 1e-12
            assert np.all(o[0, h, i, i + 1:] == 0)


def test_softcap_after_bias_order():
    # q = 0, window 3: scores are c*tanh(-slope*delta/c) for delta in {0,1,2} -> closed-form LSE; this pins
    # the order c(s + r) (bias inside the cap), not c(s) + r
    c, a, N = 0.5, 0.9, 8
    q = np.zeros((1, 1, N, 4))
    k = _rand((1, 1, N, 4), 23)
    v = _rand((1, 1, N, 4), 24)
    o, lse = orc.attention(q, k, v, CAUSAL_WIN(3), score=dict(alibi_slopes=[a], softcap=c))
    for i in range(N):
        deltas = np.arange(min(i, 2) + 1)
        inside = c * np.tanh(-a * deltas / c)
        assert abs(lse[0, 0, i] - math.log(np.exp(inside).sum())) < 1e-13
        outside = c * np.tanh(0.0) - a * deltas
        if i > 0:
            assert abs(lse[0, 0, i] - math.log(np.exp(outside).sum())) > 1e-3


def test_rel_bias_closed_form():
    N, H = 9, 2
    q = np.zeros((1, H, N, 4))
    k, v = _rand((1, H, N, 4), 25), _rand((1, H, N, 4), 26)
    rel = _rand((H, 2 * N - 1), 27)
    rule = [("window", 4), ("prefix", 2), ("or",)]
    o, lse = orc.attention(q, k, v, rule, score=dict(rel_bias=rel))
    for h in range(H):
        for i in range(N):
            js = [j for j in range(N) if (i - j < 4) or j < 2]
            want = math.log(sum(math.exp(rel[h, i - j + N - 1]) for j in js))
            assert abs(lse[0, h, i] - want) < 1e-12


def test_empty_rows_zero_output():
    q, k, v = _rand((1, 1, 6, 4), 28), _rand((1, 1, 6, 4), 29), _rand((1, 1, 6, 4), 30)
    o, lse = orc.attention(q, k, v, [("prefix", 0)])
    assert np.all(o == 0) and np.all(np.isneginf(lse))
    t = orc.block_mask([("prefix", 0)], 1, 1, 6, 6, 2, 2)
    assert not t["kv_num"].any() and not t["full_kv_num"].any()


# ------------------------------------------------------------------ split merge and paged decode
def test_split_merge_any_partition():
    rng = np.random.default_rng(31)
    s = rng.standard_normal(40) * 3
    s[[3, 17, 18]] = -np.inf
    v = rng.standard_normal((40, 5))
    m_all, l_all, u_all = orc.split_state(s, v)
    for trial in range(20):
        cuts = np.sort(rng.choice(np.arange(1, 40), size=rng.integers(1, 8), replace=False))
        parts = np.split(np.arange(40), cuts)
        st = [orc.split_state(s[p], v[p]) for p in parts]
        st.append((-np.inf, 0.0, np.zeros(5)))                       # an empty split contributes 0
        m = np.array([x[0] for x in st])
        l = np.array([x[1] for x in st])
        u = np.array([x[2] for x in st])
        o, lse = orc.merge_partials(m, l, u)
        assert np.max(np.abs(o - u_all / l_all)) < 1e-12
        assert abs(lse - (m_all + math.log(l_all))) < 1e-12


def _tiny_decode(prefix=0, seed=32):
    rng = np.random.default_rng(seed)
    Bz, Hq, Hkv, d, page, max_pages = 3, 4, 2, 8, 8, 6
    lens = np.array([13, 48, 1])
    npg = [-(-L // page) for L in lens]
    perm = rng.permutation(sum(npg))
    table = np.full((Bz, max_pages), -1, np.int32)
    p = 0
    for b in range(Bz):
        table[b, :npg[b]] = perm[p:p + npg[b]]
        p += npg[b]
    kp = rng.standard_normal((sum(npg), Hkv, page, d))
    vp = rng.standard_normal((sum(npg), Hkv, page, d))
    q = rng.standard_normal((Bz, Hq, d))
    rule = [("causal",)] if not prefix else [("causal",), ("prefix", prefix), ("or",)]
    return q, kp, vp, table, lens, rule


def test_decode_paged_equals_contiguous():
    q, kp, vp, table, lens, rule = _tiny_decode()
    o, lse = orc.decode_attention(q, kp, vp, table, lens, rule)
    for b in range(len(lens)):
        L = int(lens[b])
        kb = orc.gather_pages(kp, table, b, -(-L // 8))[:, :L]
        vb = orc.gather_pages(vp, table, b, -(-L // 8))[:, :L]
        # contiguous KV, the new token is the last position: plain softmax over all L keys
        for h in range(4):
            s = (q[b, h] @ kb[h // 2].T) / math.sqrt(8)
            p = np.exp(s - s.max())
            assert np.max(np.abs(o[b, h] - (p / p.sum()) @ vb[h // 2])) < 1e-12
            assert abs(lse[b, h] - (s.max() + math.log(p.sum()))) < 1e-12
    o2, lse2 = orc.decode_attention(q, kp, vp, table, lens[:2] * 0 + lens[:2], [("causal",), ("prefix", 1),
                                                                             ("or",)], requests=[0, 1])
    assert np.max(np.abs(o2[:2] - o[:2])) < 1e-15   # prefix region already visible -> same result


def test_decode_rejects_rules_that_see_unallocated_pages():
    q, kp, vp, table, lens, _ = _tiny_decode()
    with pytest.raises(ValueError):
        orc.decode_attention(q, kp, vp, table, lens, [("true",)])


# ------------------------------------------------------------------ planted mistakes are caught
def test_planted_mistakes_fail_pins(golden_dir, monkeypatch):
    real_allowed = orc.allowed

    def strict_causal(rule, i_g, j, dq=None, dk=None):       # plant: i > j instead of i >= j
        rule = [("window", 10**9) if op[0] == "causal" else op for op in rule]
        return real_allowed(rule, i_g, j, dq, dk) & (np.asarray(i_g) > np.asarray(j))

    monkeypatch.setattr(orc, "allowed", strict_causal)
    with pytest.raises(AssertionError):
        test_n8_w4_2x2_worked_example(golden_dir)
    monkeypatch.setattr(orc, "allowed", real_allowed)

    real_mod = orc.score_mod

    def cap_then_bias(s, h, i_g, j, score, kv_len):          # plant: c(s) + r instead of c(s + r)
        sc = dict(score or {})
        slopes = sc.pop("alibi_slopes", None)
        s = real_mod(s, h, i_g, j, sc, kv_len)
        if slopes is not None:
            s = s - float(slopes[h]) * (np.asarray(i_g) - np.asarray(j))
        return s

    monkeypatch.setattr(orc, "score_mod", cap_then_bias)
    with pytest.raises(AssertionError):
        test_softcap_after_bias_order()
    monkeypatch.setattr(orc, "score_mod", real_mod)

    real_rows = orc.attention_rows

    def unscaled(q_rows, k, v, rule, rows, b, h, q_len, kv_len, scale, *a, **kw):   # plant: drop the scale
        return real_rows(q_rows, k, v, rule, rows, b, h, q_len, kv_len, 1.0, *a, **kw)

    monkeypatch.setattr(orc, "attention_rows", unscaled)
    with pytest.raises(AssertionError):
        test_matches_torch_sdpa_fp64(True)


# ------------------------------------------------------------------ backward
def _finite_difference_check(rule, score, B=1, Hq=2, Hkv=1, N=11, d=6, doc=None, seed=0, samples=6):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hq, N, d))
    k = rng.standard_normal((B, Hkv, N, d))
    v = rng.standard_normal((B, Hkv, N, d))
    do = rng.standard_normal((B, Hq, N, d))
    dq, dk, dv = orc.attention_backward(q, k, v, do, rule, None, score, doc_ids=doc)

    def loss(q_, k_, v_):
        o, _ = orc.attention(q_, k_, v_, rule, None, score, doc_ids=doc)
        return float(np.sum(o * do))

    eps = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(samples):
            idx = tuple(int(rng.integers(0, n)) for n in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - grad[idx]) < 1e-6 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


@pytest.mark.parametrize("case", ["causal_window_softcap_alibi", "doc_prefix", "dense_gqa", "empty_rows"])
def test_backward_matches_finite_differences(case):
    # central differences of L = sum(O * dO) (brute force, independent of the gradient formulas)
    if case == "causal_window_softcap_alibi":
        _finite_difference_check([("causal",), ("window", 5), ("and",)], {"softcap": 3.0, "alibi_slopes": [0.5, 0.25]})
    elif case == "doc_prefix":
        doc = np.array([[0, 0, 0, 1, 1, 1, 1, 2, 2, 2, 2]], dtype=np.int32)
        _finite_difference_check([("causal",), ("prefix", 2), ("or",), ("doc",), ("and",)], None, doc=doc, seed=1)
    elif case == "dense_gqa":
        _finite_difference_check([("true",)], None, Hq=4, Hkv=2, seed=2)
    else:  # rows that see nothing carry no gradient, and nothing flows to the keys they cannot see
        _finite_difference_check([("prefix", 0)], None, seed=3)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_torch_autograd(causal):
    # the same gradients from torch's autograd of torch.softmax on fp64 tensors (a library routine)
    rng = np.random.default_rng(7 + causal)
    B, Hq, Hkv, N, d = 2, 4, 2, 9, 8
    q = rng.standard_normal((B, Hq, N, d))
    k = rng.standard_normal((B, Hkv, N, d))
    v = rng.standard_normal((B, Hkv, N, d))
    do = rng.standard_normal((B, Hq, N, d))
    rule = [("causal",)] if causal else [("true",)]
    dq, dk, dv = orc.attention_backward(q, k, v, do, rule, 0.3, {"softcap": 2.5})
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    ke, ve = tk.repeat_interleave(Hq // Hkv, dim=1), tv.repeat_interleave(Hq // Hkv, dim=1)
    s = 2.5 * torch.tanh(0.3 * (tq @ ke.transpose(-1, -2)) / 2.5)
    if causal:
        s = s.masked_fill(~torch.ones(N, N, dtype=torch.bool).tril(), float("-inf"))
    o = torch.softmax(s, dim=-1) @ ve
    gq, gk, gv = torch.autograd.grad(o, (tq, tk, tv), torch.tensor(do))
    np.testing.assert_allclose(dq, gq.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, gk.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, gv.numpy(), atol=1e-12)


def test_planted_backward_mistake_is_caught(monkeypatch):
    real = orc.attention_backward

    def no_cap_derivative(q, k, v, do, rule, scale=None, score=None, q_offset=None, doc_ids=None):
        # plant: the soft-cap chain-rule factor dropped (gradient taken as if s' = s)
        rng_q, rng_k, rng_v = real(q, k, v, do, rule, scale, None, q_offset, doc_ids)
        return rng_q, rng_k, rng_v

    monkeypatch.setattr(orc, "attention_backward", no_cap_derivative)
    with pytest.raises(AssertionError):
        test_backward_matches_torch_autograd(False)
