"""fa_flex_backward on the GPU vs the fp64 oracle's gradients on the same bf16 inputs: dQ, dK, dV over
masks with windows, prefixes, documents, GQA, soft-cap and ALiBi, ragged lengths, empty rows.

Tolerance (derived from the arithmetic): P and dS enter the tensor-core products as bf16 (relative
rounding <= 2^-8 per element) with fp32 accumulation, and the forward's fp32 O enters D; for a gradient
tensor g with scale G = max|g*| the error bound used is max|g - g*| <= 2e-2 G and mean|g - g*| <= 2e-3 G."""
import math

import numpy as np
import pytest
import torch

from block_sparse_masked_create_gb300 import fa, synth, workloads
from oracle import flexmask_oracle as orc
from tests import gpu_common as gc

pytestmark = pytest.mark.gpu

G_MAX, G_MEAN = 2e-2, 2e-3


def case(name, B, Hq, Hkv, q_len, kv_len, d, bq, bk, rule, score=None, doc=None, seed=21):
    w = workloads.Prefill(name, B, Hq, Hkv, q_len, kv_len, d, bq, bk, rule, score or {}, 1.0 / math.sqrt(d), seed)
    if doc is not None:
        w.doc_ids = doc
    return w.generate()


def run_backward(w):
    r = gc.run_prefill(w, out_dtype=torch.float32)
    assert r["status"] == fa.OK
    al, rb, doc, q, k, v = r["keep"]
    sc = fa.make_score_rule(al, rb, w.score.get("softcap", 0.0))  # the forward's bias tensors, still alive
    dout = workloads.bf16_torch(w.dout_bits(), "cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dq, dk, dv = fa.flex_backward(q, k, v, r["out"], r["lse"], dout, r["bm"], sc, w.scale, status=status)
    assert fa.check_status(status) == fa.OK
    return dq.cpu().numpy(), dk.cpu().numpy(), dv.cpu().numpy()


def oracle_grads(w):
    qf, kf, vf, df = (synth.bf16_bits_to_f64(x) for x in (w.q_bits, w.k_bits, w.v_bits, w.dout_bits()))
    return orc.attention_backward(qf, kf, vf, df, w.rule, w.scale, gc.oracle_score(w.score), doc_ids=w.doc_ids)


def check(w):
    got = run_backward(w)
    want = oracle_grads(w)
    for name, g, r in zip(("dq", "dk", "dv"), got, want):
        G = max(float(np.abs(r).max()), 1e-6)
        err = np.abs(g - r)
        print(f"{w.name} {name}: max {err.max():.3e} mean {err.mean():.3e} scale {G:.3e}")
        assert np.all(np.isfinite(g)), f"{w.name} {name}: non-finite"
        assert err.max() <= G_MAX * G, f"{w.name} {name}: max err {err.max():.3e} > {G_MAX} x {G:.3e}"
        assert err.mean() <= G_MEAN * G, f"{w.name} {name}: mean err {err.mean():.3e} > {G_MEAN} x {G:.3e}"


CW = lambda w: [("causal",), ("window", w), ("and",)]
DOCS = np.repeat(np.arange(6, dtype=np.int32), [70, 30, 100, 20, 60, 40])[None, :]


@pytest.mark.parametrize("cfg", [
    ("causal_d64_64x64", 1, 2, 2, 256, 256, 64, 64, 64, [("causal",)], None),
    ("causal_d128_128x128", 1, 2, 2, 384, 384, 128, 128, 128, [("causal",)], None),
    ("window_softcap_gqa", 2, 4, 2, 320, 320, 128, 128, 128, CW(100), {"softcap": 20.0}),
    ("dense_64x128", 1, 2, 1, 192, 256, 64, 64, 128, [("true",)], None),
    ("prefix_or_causal_128x64", 1, 2, 2, 256, 256, 128, 128, 64, [("causal",), ("prefix", 40), ("or",)], None),
    ("ragged", 1, 2, 2, 200, 200, 128, 128, 128, [("causal",)], None),
    ("causal_d64_128x128", 1, 2, 1, 384, 384, 64, 128, 128, [("causal",)], None),
    ("window_gqa_ragged_128", 2, 4, 1, 300, 300, 128, 128, 128, CW(150), None),
    ("dense_rect_128", 1, 2, 2, 192, 320, 128, 128, 128, [("true",)], None),
    ("prefix_or_window_softcap_d64_128", 1, 2, 2, 400, 400, 64, 128, 128,
     [("causal",), ("window", 90), ("and",), ("prefix", 30), ("or",)], {"softcap": 30.0}),
])
def test_backward_small(cfg):
    name, B, Hq, Hkv, ql, kl, d, bq, bk, rule, score = cfg
    check(case(name, B, Hq, Hkv, ql, kl, d, bq, bk, rule, score))


def test_backward_documents_alibi():
    slopes = [2.0 ** (-8.0 * (h + 1) / 4) for h in range(4)]
    w = case("doc_alibi", 1, 4, 2, 320, 320, 128, 128, 128, [("causal",), ("doc",), ("and",)],
             {"alibi_slopes": slopes}, doc=DOCS)
    check(w)


def test_backward_unseen_keys_have_zero_gradient():
    # keys >= 64 are never allowed (causal and a 64-key prefix): their dK, dV rows are exactly zero
    w = case("unseen_keys", 1, 2, 2, 256, 256, 64, 64, 64, [("causal",), ("prefix", 64), ("and",)])
    dq, dk, dv = run_backward(w)
    want = oracle_grads(w)
    for g, r in zip((dq, dk, dv), want):
        G = max(float(np.abs(r).max()), 1e-6)
        assert np.abs(g - r).max() <= G_MAX * G
    assert np.abs(dk[:, :, 64:]).max() == 0.0 and np.abs(dv[:, :, 64:]).max() == 0.0


@pytest.mark.parametrize("blk", [64, 128])
def test_backward_empty_rows_give_zero(blk):
    # no pair allowed at all: every row is empty (O = 0, LSE = -inf) and every gradient is exactly zero
    w = case("all_empty", 1, 2, 1, 130, 130, 64, blk, blk, [("prefix", 0)])
    dq, dk, dv = run_backward(w)
    assert np.abs(dq).max() == 0.0 and np.abs(dk).max() == 0.0 and np.abs(dv).max() == 0.0


def test_backward_unseen_key_blocks_128():
    # 128x128 blocks: key blocks 1 and 2 are never visited (causal and a 128-key prefix), so their CTAs
    # have no query block to walk and write zero dK, dV
    w = case("unseen_blocks", 1, 2, 1, 384, 384, 128, 128, 128, [("causal",), ("prefix", 128), ("and",)])
    dq, dk, dv = run_backward(w)
    want = oracle_grads(w)
    for g, r in zip((dq, dk, dv), want):
        G = max(float(np.abs(r).max()), 1e-6)
        assert np.abs(g - r).max() <= G_MAX * G
    assert np.abs(dk[:, :, 128:]).max() == 0.0 and np.abs(dv[:, :, 128:]).max() == 0.0


def test_backward_cfg2_shape_sampled_heads():
    # the causal workload's block geometry at reduced batch (B=1, 2 heads, N=2048): full oracle gradients
    w = workloads.cfg2(B=1, H=2, n=2048).generate()
    check(w)


@pytest.mark.parametrize("kind", ["unsorted", "sorted_with_minus_one"])
def test_backward_documents_id_orders(kind):
    # document equality from id runs (ids that never decrease) and from id-by-id comparison (any order;
    # -1 ids, which positions outside the id array also read), on 128x128 blocks with GQA
    rng = np.random.default_rng(91 if kind == "unsorted" else 92)
    n = 384
    ids = rng.integers(-1 if kind != "unsorted" else 0, 4, size=n).astype(np.int32)
    if kind != "unsorted":
        ids = np.sort(ids)
    w = case(f"doc_{kind}", 1, 4, 2, n, n, 128, 128, 128, [("causal",), ("doc",), ("and",)], None, doc=ids[None, :])
    check(w)


def test_backward_cfg2_full_size_sampled_heads():
    # the benchmarked configuration itself (B=4, H=16, N=4096, d=128, causal), run whole on the GPU; two
    # seeded (b, h) pairs checked against the oracle on that head alone (one KV head per query head, so a
    # head is an independent problem)
    w = workloads.cfg2().generate()
    dq, dk, dv = run_backward(w)
    rng = np.random.default_rng(5)
    pairs = [(0, 0), (int(rng.integers(w.B)), int(rng.integers(w.Hq)))]
    do = w.dout_bits()
    for b, h in pairs:
        f = lambda x: synth.bf16_bits_to_f64(x[b:b + 1, h:h + 1])
        want = orc.attention_backward(f(w.q_bits), f(w.k_bits), f(w.v_bits), f(do), w.rule, w.scale)
        for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), want):
            g = g[b:b + 1, h:h + 1]
            G = max(float(np.abs(r).max()), 1e-6)
            err = np.abs(g - r)
            assert err.max() <= G_MAX * G, f"({b},{h}) {name}: max err {err.max():.3e} > {G_MAX} x {G:.3e}"
            assert err.mean() <= G_MEAN * G, f"({b},{h}) {name}: mean err {err.mean():.3e}"
