"""fa_flex_forward on the GPU vs the fp64 oracle on the same seeded bf16 inputs.

Small cases compare every output element (ragged tails, several tiles, all rule atoms and their
compositions, every score rule, MHA/GQA/MQA, empty rows, large scores); the workloads run at their full
size in the launch configuration the benchmark times and are compared on sampled rows. Both kernels
(tcgen05 for 128x128 blocks, mma.sync for the rest and as a cross-check) are exercised.
Tolerances: max |O err| <= 8e-3, mean |O err| <= 1e-3, max |LSE err| <= 2e-3."""
import math

import numpy as np
import pytest
import torch

from block_sparse_masked_create_gb300 import fa, synth, workloads
from oracle import flexmask_oracle as orc
from tests import gpu_common as gc

pytestmark = pytest.mark.gpu

CW = lambda w: [("causal",), ("window", w), ("and",)]


def small(name, B, Hq, Hkv, q_len, kv_len, d, bq, bk, rule, score=None, scale=None, doc=None, seed=7):
    w = workloads.Prefill(name, B, Hq, Hkv, q_len, kv_len, d, bq, bk, rule, score or {},
                          scale if scale else 1.0 / math.sqrt(d), seed)
    if doc is not None:
        w.doc_ids = doc
    return w.generate()


def full_compare(w, force_mma=False, what="", out_dtype=torch.float32):
    r = gc.run_prefill(w, force_mma=force_mma, out_dtype=out_dtype)
    assert r["status"] == fa.OK
    assert r["out"].dtype == out_dtype
    o = r["out"].float().cpu().numpy()
    lse = r["lse"].cpu().numpy()
    qf, kf, vf = (synth.bf16_bits_to_f64(x) for x in (w.q_bits, w.k_bits, w.v_bits))
    o_ref, lse_ref = orc.attention(qf, kf, vf, w.rule, w.scale, gc.oracle_score(w.score), doc_ids=w.doc_ids)
    return gc.compare(o, lse, o_ref, lse_ref, what or w.name, out_bf16=out_dtype == torch.bfloat16), r


DOC = np.repeat(np.arange(7, dtype=np.int32), [40, 3, 100, 17, 60, 9, 200])[None, :]


CASES = [
    # name, B, Hq, Hkv, q_len, kv_len, d, bq, bk, rule, score
    ("causal_ragged", 2, 2, 1, 300, 300, 128, 128, 128, [("causal",)], {}),
    ("window_gqa_softcap", 1, 4, 2, 512, 512, 64, 64, 64, CW(128), dict(softcap=20.0)),
    ("cross_len", 1, 2, 2, 200, 333, 128, 64, 32, [("true",)], {}),
    ("prefix_or", 1, 3, 1, 257, 257, 64, 32, 64, [("causal",), ("prefix", 70), ("or",)], {}),
    ("doc_alibi", 1, 4, 4, 429, 429, 128, 128, 128, [("causal",), ("doc",), ("and",)],
     dict(alibi_slopes=workloads.alibi_slopes(4))),
    ("window_softcap_128", 1, 2, 2, 700, 700, 128, 128, 128, CW(200), dict(softcap=30.0)),
    ("relbias_tiny", 1, 2, 1, 70, 70, 64, 16, 16, CW(33), None),
    ("bias_then_cap", 1, 2, 2, 150, 150, 64, 32, 32, [("causal",)],
     dict(alibi_slopes=np.array([0.05, 0.3], np.float32), softcap=5.0)),
    ("mqa_block16", 1, 4, 1, 96, 96, 128, 16, 128, CW(40), {}),
    # more (batch, head pair) units than one group of eight, on the 128x128 path: the group order of the
    # tcgen05 kernel (two tiles per CTA; one tile per CTA for the MHA window) is checked on every element
    ("causal_9_pairs", 3, 6, 6, 384, 384, 128, 128, 128, [("causal",)], {}),
    ("gqa_12_pairs_softcap", 2, 12, 4, 384, 384, 128, 128, 128, CW(200), dict(softcap=30.0)),
    ("window_mha_10_heads", 2, 5, 5, 512, 512, 128, 128, 128, CW(256), {}),
    # soft-cap with the fixed reference maximum: rows that see no key at all (queries past the keys' window)
    # must still come out empty; a cap too large for the fixed reference (c log2(e) > 90) takes the
    # generic score path
    ("softcap_empty_rows", 1, 2, 2, 300, 100, 128, 128, 128, [("window", 50)], dict(softcap=30.0)),
    ("softcap_large_cap", 1, 2, 2, 400, 400, 128, 128, 128, CW(200), dict(softcap=80.0)),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("force_mma", [False, True])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_small_cases_all_elements(case, force_mma, out_dtype):
    name, B, Hq, Hkv, ql, kl, d, bq, bk, rule, score = case
    if score is None:  # relative-bias table
        rng = np.random.default_rng(3)
        score = dict(rel_bias=(rng.standard_normal((Hq, 2 * kl - 1)) * 2).astype(np.float32))
    doc = DOC[:, :max(ql, kl)] if any(op[0] == "doc" for op in rule) else None
    w = small(name, B, Hq, Hkv, ql, kl, d, bq, bk, rule, score, doc=doc)
    full_compare(w, force_mma=force_mma, out_dtype=out_dtype)


def test_empty_rows_and_no_loads():
    w = small("empty", 1, 2, 2, 130, 130, 128, 128, 128, [("prefix", 0)])
    r = gc.run_prefill(w, counters=True)
    assert r["status"] == fa.OK
    assert torch.all(r["out"] == 0) and torch.all(torch.isneginf(r["lse"]))
    c = r["counters"].cpu().tolist()
    assert c[1] == 0 and c[2] == 0 and c[3] == 0          # no block visited, no K/V tile loaded


def test_partially_empty_rows():
    # cross attention, q_len > kv_len with a causal window: rows i >= kv_len - 1 + W see no key at all
    w = small("part_empty", 1, 2, 1, 256, 100, 64, 64, 32, CW(30))
    errs, r = full_compare(w)
    assert torch.all(torch.isneginf(r["lse"][:, :, 129:])) and torch.all(r["out"][:, :, 129:] == 0)


def test_large_scores():
    w = small("large", 1, 2, 2, 256, 256, 128, 128, 128, [("causal",)])
    qb = synth.bf16_bits_to_f64(w.q_bits) * 12.0                  # scores of order +-100
    w.q_bits = np.vectorize(synth.bf16_bits_from_double, otypes=[np.uint16])(qb)
    full_compare(w)


@pytest.mark.parametrize("name", ["cfg1"])
def test_cfg1_all_elements(name):
    w = workloads.cfg1().generate()
    errs, r = full_compare(w)
    errs2, _ = full_compare(w, force_mma=True)
    errs3, _ = full_compare(w, out_dtype=torch.bfloat16)


@pytest.mark.parametrize("name", ["cfg2", "cfg3", "cfg4"])
def test_full_size_sampled(name):
    # the launch configuration the benchmark times (fp32 O); every (b, h) pair, and from every query block
    # (each holds a partial block) its first, last and one random row
    w = {"cfg2": workloads.cfg2, "cfg3": workloads.cfg3, "cfg4": workloads.cfg4}[name]().generate()
    r = gc.run_prefill(w, counters=True)
    assert r["status"] == fa.OK
    per_block = gc.sample_rows_every_block(w, seed=11)
    rows = np.concatenate([np.asarray(x, dtype=np.int64) for x in per_block])
    out, lse = r["out"], r["lse"]
    assert out.dtype == torch.float32
    ridx = torch.from_numpy(rows).cuda()
    o_all = out[:, :, ridx].cpu().numpy()
    l_all = lse[:, :, ridx].cpu().numpy()
    for b in range(w.B):
        for h in range(w.Hq):
            o_ref, lse_ref = gc.oracle_rows_per_block(w, b, h, per_block)
            gc.compare(o_all[b, h], l_all[b, h], o_ref, lse_ref, f"{name} b={b} h={h}")
    # counters: every visited block of every tile counted once; a CTA's two tiles read one KV head and load
    # each block of the union of their lists once (K and V), so the loads lie between one and two per
    # visited tile-block
    st = fa.block_mask_stats(r["bm"]).cpu().tolist()
    c = r["counters"].cpu().tolist()
    heads = w.B * w.Hq // (r["bm"].c.Bm * r["bm"].c.Hm)
    assert c[1] == st[0] * heads and c[2] == st[1] * heads
    visited = c[1] + c[2]
    assert visited <= c[3] <= 2 * visited
    assert np.all(np.isfinite(out.float().cpu().numpy()))


def test_tc5_and_mma_kernels_cfg2_small_against_oracle():
    # both kernels on a reduced cfg2 (B=1, H=4, N=1024), every element against the oracle
    w = workloads.cfg2(B=1, H=4, n=1024).generate()
    full_compare(w, what="cfg2 small tcgen05")
    full_compare(w, force_mma=True, what="cfg2 small mma.sync")


@pytest.mark.parametrize("kind", ["causal_mha", "gqa_docs_per_batch_alibi", "head_dependent_window_bf16"])
def test_forward_from_host_buffers(kind):
    # fa_flex_forward_host streams chunks of KV heads through two device slots: bit-identical to the
    # device forward, with per-batch document ids and query offsets, per-head tables and per-head ALiBi
    # slopes taken at each chunk's offsets
    dev = "cuda"
    if kind == "causal_mha":
        w = workloads.cfg2(B=2, H=6, n=640).generate()
        doc = off = None
        out_dtype, hdep = torch.float32, False
    elif kind == "gqa_docs_per_batch_alibi":
        w = workloads.Prefill("host_gqa", 3, 8, 2, 384, 384, 128, 128, 128, [("causal",), ("doc",), ("and",)],
                              {"alibi_slopes": [2.0 ** (-(h + 1)) for h in range(8)]}, 1.0 / math.sqrt(128), 77)
        w.generate()
        rng = np.random.default_rng(3)
        doc = np.sort(rng.integers(0, 5, size=(3, 384)), axis=1).astype(np.int32)
        off = None
        out_dtype, hdep = torch.float32, False
    else:
        w = workloads.Prefill("host_hdep", 1, 4, 4, 500, 500, 64, 128, 128, [("causal",), ("window", 200), ("and",)],
                              {}, 1.0 / math.sqrt(64), 78)
        w.generate()
        doc = off = None
        out_dtype, hdep = torch.bfloat16, True
    doc_t = None if doc is None else torch.from_numpy(doc).to(dev)
    rule = fa.make_mask_rule(w.rule, doc_ids=doc_t, head_dependent=hdep)
    bm = fa.create_block_mask(rule, w.B, w.Hq, w.q_len, w.kv_len, w.bq, w.bk, device=dev, keep=[doc_t])
    al, rb, sc = gc.score_tensors(w.score, dev)
    q = workloads.bf16_torch(w.q_bits, dev)
    k = workloads.bf16_torch(w.k_bits, dev)
    v = workloads.bf16_torch(w.v_bits, dev)
    o_dev, l_dev = fa.flex_forward(q, k, v, bm, sc, w.scale, out_dtype=out_dtype)
    hq = workloads.bf16_torch(w.q_bits).pin_memory()
    hk = workloads.bf16_torch(w.k_bits).pin_memory()
    hv = workloads.bf16_torch(w.v_bits).pin_memory()
    ho = torch.empty(q.shape, dtype=out_dtype).pin_memory()
    hl = torch.empty((w.B, w.Hq, w.q_len), dtype=torch.float32).pin_memory()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    fa.flex_forward_host(hq, hk, hv, bm, sc, w.scale, out=ho, lse=hl, status=status)
    torch.cuda.synchronize()
    assert fa.check_status(status) == fa.OK
    assert torch.equal(ho.view(torch.int16 if out_dtype == torch.bfloat16 else torch.int32),
                       o_dev.cpu().view(torch.int16 if out_dtype == torch.bfloat16 else torch.int32))
    assert torch.equal(hl.view(torch.int32), l_dev.cpu().view(torch.int32))
