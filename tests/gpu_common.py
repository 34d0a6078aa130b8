"""Shared helpers of the GPU parity tests: run the library through the C ABI on seeded inputs and compare
with the fp64 oracle on the same inputs (full tensors for small cases, sampled rows at full size)."""
from __future__ import annotations

import numpy as np
import torch

from block_sparse_masked_create_gb300 import fa, synth, workloads
from oracle import flexmask_oracle as orc

# bf16 inputs, fp32 accumulation, fp64 reference (tolerances fixed by the target specification)
O_MAX, O_MEAN, LSE_MAX = 8e-3, 1e-3, 2e-3


def rule_arrays(w: workloads.Prefill, device="cuda"):
    doc = None if w.doc_ids is None else torch.from_numpy(np.ascontiguousarray(w.doc_ids.astype(np.int32))).to(device)
    return doc


def score_tensors(score: dict, device="cuda"):
    al = score.get("alibi_slopes")
    rb = score.get("rel_bias")
    al_t = None if al is None else torch.tensor(np.asarray(al, dtype=np.float32), device=device)
    rb_t = None if rb is None else torch.from_numpy(np.ascontiguousarray(np.asarray(rb, dtype=np.float32))).to(device)
    return al_t, rb_t, fa.make_score_rule(al_t, rb_t, score.get("softcap", 0.0))


def oracle_score(score: dict) -> dict:
    out = {}
    if score.get("alibi_slopes") is not None:
        out["alibi_slopes"] = np.asarray(score["alibi_slopes"], dtype=np.float32).astype(np.float64)
    if score.get("rel_bias") is not None:
        out["rel_bias"] = np.asarray(score["rel_bias"], dtype=np.float32).astype(np.float64)
    if score.get("softcap"):
        out["softcap"] = float(score["softcap"])
    return out


def run_prefill(w: workloads.Prefill, force_mma=False, counters=False, bq=None, bk=None, out_dtype=torch.float32):
    """Generate (if needed) and run create_block_mask + flex_forward; returns dict of results."""
    if w.q_bits is None:
        w.generate()
    dev = "cuda"
    q = workloads.bf16_torch(w.q_bits, dev)
    k = workloads.bf16_torch(w.k_bits, dev)
    v = workloads.bf16_torch(w.v_bits, dev)
    doc = rule_arrays(w, dev)
    rule = fa.make_mask_rule(w.rule, doc_ids=doc)
    bm = fa.create_block_mask(rule, w.B, w.Hq, w.q_len, w.kv_len, bq or w.bq, bk or w.bk, device=dev, keep=[doc])
    al, rb, sc = score_tensors(w.score, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    cnt = torch.zeros(4, dtype=torch.int64, device=dev) if counters else None
    out, lse = fa.flex_forward(q, k, v, bm, sc, w.scale, status=status, counters=cnt, force_mma=force_mma,
                               out_dtype=out_dtype)
    st = fa.check_status(status)
    return dict(out=out, lse=lse, bm=bm, status=st, counters=cnt, keep=(al, rb, doc, q, k, v))


def sample_rows_every_block(w: workloads.Prefill, seed=0):
    """Seeded rows for the full-size comparison: from EVERY query block, its first and last row and one
    random row in between (every block of the prefill workloads holds a partial block: the diagonal)."""
    rng = np.random.default_rng(seed)
    nq = -(-w.q_len // w.bq)
    per_block = []
    for r in range(nq):
        lo, hi = r * w.bq, min(w.q_len, (r + 1) * w.bq)
        per_block.append(sorted({lo, hi - 1, int(rng.integers(lo, hi))}))
    return per_block


def oracle_rows_per_block(w: workloads.Prefill, b: int, h: int, per_block):
    """fp64 oracle O/LSE of one (b, h) for the rows of `per_block` (one oracle call per query block, so the
    keys no sampled row of the block may see drop out of its dot products)."""
    g = w.Hq // w.Hkv
    hk = h // g
    kf = synth.bf16_bits_to_f64(w.k_bits[b, hk])
    vf = synth.bf16_bits_to_f64(w.v_bits[b, hk])
    sc = oracle_score(w.score)
    os_, ls_ = [], []
    for rows in per_block:
        rows = np.asarray(rows, dtype=np.int64)
        qf = synth.bf16_bits_to_f64(w.q_bits[b, h, rows])
        o, l = orc.attention_rows(qf, kf, vf, w.rule, rows, b, h, w.q_len, w.kv_len, w.scale, sc, 0, w.doc_ids)
        os_.append(o)
        ls_.append(l)
    return np.concatenate(os_), np.concatenate(ls_)


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Half a bf16 ulp at |x| (8 significant bits): the largest error of rounding x to bf16."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, np.ldexp(1.0, (e - 8).astype(np.int64)), 0.0)


def compare(o_gpu: np.ndarray, lse_gpu: np.ndarray, o_ref: np.ndarray, lse_ref: np.ndarray, what="",
            out_bf16: bool = False):
    """Tolerance check: max/mean |O - O*| and max |LSE - LSE*| (empty rows: LSE both -inf, O both 0).

    fp32 output: the bounds apply as stated. bf16 output: the stored value also carries the rounding of
    the result to bf16, at most half an ulp of O*, which is added to the max bound element by element (the
    max bound alone is below that rounding for |O*| >= 4); the mean bound stays 1e-3 as stated."""
    err = np.abs(o_gpu.astype(np.float64) - o_ref)
    slack = half_ulp_bf16(o_ref) if out_bf16 else np.zeros_like(o_ref)
    inf_ref = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse_gpu), inf_ref), f"{what}: empty-row pattern differs"
    lerr = np.abs(lse_gpu[~inf_ref].astype(np.float64) - lse_ref[~inf_ref]) if (~inf_ref).any() else np.zeros(1)
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite output"
    assert np.all(err <= O_MAX + slack), f"{what}: max |O err| {err.max():.3e} (excess {(err - slack).max():.3e})"
    assert err.mean() <= O_MEAN, f"{what}: mean |O err| {err.mean():.3e}"
    assert lerr.max() <= LSE_MAX, f"{what}: max |LSE err| {lerr.max():.3e}"
    return float(err.max()), float(err.mean()), float(lerr.max())


def tables_np(bm: fa.BlockMask) -> dict:
    t = bm.tables()
    return {k: v.cpu().numpy() for k, v in t.items()}


def assert_row_order(got: dict, want: dict):
    """The builder's row order: query block rows by visited length (full + partial) from the longest, ties
    by the higher row first; derived here from the oracle's tables with a stable sort."""
    ln = want["kv_num"] + want["full_kv_num"]                        # [Bm, Hm, nq]
    nq = ln.shape[2]
    if nq == 1:                                                      # nothing to order: no table
        assert "row_order" not in got
        return
    rows_desc = np.arange(nq - 1, -1, -1)
    if want["nk"] > 2048:                                            # wide tables keep nq-1 .. 0
        assert (got["row_order"] == rows_desc).all()
        return
    for bm in range(ln.shape[0]):
        for hm in range(ln.shape[1]):
            l_desc = ln[bm, hm, rows_desc]
            expect = rows_desc[np.argsort(-l_desc, kind="stable")]
            assert np.array_equal(got["row_order"][bm, hm], expect), f"row order ({bm},{hm})"


def assert_tables_equal(got: dict, want: dict, rows=None):
    keys = ["kv_num", "kv_idx", "full_kv_num", "full_kv_idx", "block_class"]
    for k in keys:
        g, w_ = got[k], want[k]
        if rows is not None:
            g, w_ = g[:, :, rows], w_[:, :, rows]
        assert g.shape == w_.shape, f"{k}: shape {g.shape} vs {w_.shape}"
        assert np.array_equal(g, w_), f"{k}: tables differ"
    if rows is None:
        for k in ["q_num", "q_idx", "full_q_num", "full_q_idx"]:
            assert np.array_equal(got[k], want[k]), f"{k}: tables differ"
