"""fa_flex_decode (paged split-KV) on the GPU vs the fp64 paged oracle on the same seeded inputs: small
cases on every element, the 64-request workload at full size on every request and head, and the
device-side page-id check."""
import math

import numpy as np
import pytest
import torch

from block_sparse_masked_create_gb300 import fa, synth, workloads
from oracle import flexmask_oracle as orc
from tests import gpu_common as gc

pytestmark = pytest.mark.gpu


def run_decode(d: workloads.Decode, table=None, out_dtype=torch.float32):
    dev = "cuda"
    q = workloads.bf16_torch(d.q_bits, dev)
    kp = workloads.bf16_torch(d.k_bits, dev)
    vp = workloads.bf16_torch(d.v_bits, dev)
    pt = torch.from_numpy(np.ascontiguousarray(d.page_table if table is None else table)).to(dev)
    off = torch.from_numpy(d.q_offset).to(dev)
    rule = fa.make_mask_rule(d.rule, q_offset=off, batch_dependent=True)
    bm = fa.create_block_mask(rule, d.Bz, d.Hq, 1, d.kv_len, 1, d.page, keep=[off])
    al, rb, sc = gc.score_tensors(d.score, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    cnt = torch.zeros(4, dtype=torch.int64, device=dev)
    out, lse = fa.flex_decode(q, kp, vp, pt, bm, sc, d.scale, status=status, counters=cnt, out_dtype=out_dtype)
    st = fa.check_status(status)
    return out, lse, st, cnt


def oracle_decode(d, requests):
    q = synth.bf16_bits_to_f64(d.q_bits)
    kp = synth.bf16_bits_to_f64(d.k_bits)
    vp = synth.bf16_bits_to_f64(d.v_bits)
    return orc.decode_attention(q, kp, vp, d.page_table, d.kv_lens, d.rule, d.scale, gc.oracle_score(d.score),
                                requests=requests, kv_len_table=d.kv_len)


@pytest.mark.parametrize("page,g,d_,prefix", [(128, 4, 128, 0), (32, 2, 64, 0), (64, 8, 128, 40), (32, 1, 64, 0),
                                              (128, 16, 128, 0)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_small_decode(page, g, d_, prefix, out_dtype):
    Hkv = 2
    dec = workloads.cfg5(Bz=5, Hq=Hkv * g, Hkv=Hkv, d=d_, page=page, lo=max(1, prefix), hi=9 * page + 5,
                         prefix=prefix)
    dec.generate()
    out, lse, st, cnt = run_decode(dec, out_dtype=out_dtype)
    assert st == fa.OK
    reqs = list(range(dec.Bz))
    o_ref, lse_ref = oracle_decode(dec, reqs)
    gc.compare(out.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, f"decode page={page} g={g}",
               out_bf16=out_dtype == torch.bfloat16)
    pages = sum(-(-int(L) // page) for L in dec.kv_lens)
    assert cnt.cpu().tolist()[3] == 2 * pages * Hkv            # each visited page read once per KV head


def test_decode_with_scores():
    dec = workloads.cfg5(Bz=3, Hq=8, Hkv=2, d=128, page=64, lo=100, hi=700)
    dec.score = dict(alibi_slopes=workloads.alibi_slopes(8), softcap=15.0)
    dec.generate()
    out, lse, st, _ = run_decode(dec)
    assert st == fa.OK
    o_ref, lse_ref = oracle_decode(dec, [0, 1, 2])
    gc.compare(out.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "decode scores")


def test_cfg5_full_size_every_request():
    dec = workloads.cfg5().generate()
    out, lse, st, cnt = run_decode(dec)
    assert st == fa.OK
    L = dec.kv_lens
    reqs = list(range(dec.Bz))                                  # every request, every query head
    o_ref, lse_ref = oracle_decode(dec, reqs)
    gc.compare(out.float().cpu().numpy()[reqs], lse.cpu().numpy()[reqs], o_ref[reqs], lse_ref[reqs], "cfg5")
    assert np.all(np.isfinite(out.float().cpu().numpy()))
    assert cnt.cpu().tolist()[3] == 2 * int(sum(-(-int(x) // 128) for x in L)) * dec.Hkv


def test_bad_page_id_reported():
    dec = workloads.cfg5(Bz=2, Hq=4, Hkv=2, d=64, page=32, lo=40, hi=200).generate()
    table = dec.page_table.copy()
    table[1, 0] = dec.n_pages_total + 5                      # out of range: reported, page skipped
    _, _, st, _ = run_decode(dec, table)
    assert st == fa.ERR_DEVICE_CHECK


@pytest.mark.parametrize("page,bq,kind", [(128, 128, "causal"), (64, 128, "window"), (32, 64, "prefix"),
                                          (128, 16, "window"), (64, 128, "doc")])
def test_prebuilt_mask_sliced_per_step(page, bq, kind):
    # the table is built once for the longest context in global positions; each step takes, per request,
    # the query-block row that holds the request's position and re-evaluates that row's partial blocks at
    # the position: the result must equal the one-row table built directly, and the decode over it the
    # oracle
    prefix = 40 if kind == "prefix" else 0
    dec = workloads.cfg5(Bz=6, Hq=8, Hkv=2, d=128, page=page, lo=max(1, prefix), hi=9 * page + 5, prefix=prefix)
    if kind == "window":
        dec.rule = [("causal",), ("window", 3 * page + 7), ("and",)]
    dev = "cuda"
    L = dec.kv_len
    doc = None
    if kind == "doc":
        dec.rule = [("causal",), ("doc",), ("and",)]
        ids = np.repeat(np.arange(L // 50 + 1, dtype=np.int32), 50)[:L][None, :]
        doc = torch.from_numpy(ids).to(dev)
    dec.generate()
    big = fa.create_block_mask(fa.make_mask_rule(dec.rule, doc_ids=doc), 1, dec.Hq, L, L, bq, page, keep=[doc])
    qpos = torch.from_numpy(dec.q_offset).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sel = fa.select_rows(big, qpos, status=status)
    assert sel.shape == (dec.Bz, 1, 1, dec.max_pages)
    direct = fa.create_block_mask(fa.make_mask_rule(dec.rule, doc_ids=doc, q_offset=qpos, batch_dependent=True),
                                  dec.Bz, dec.Hq, 1, L, 1, page, keep=[doc, qpos])
    ts, td = gc.tables_np(sel), gc.tables_np(direct)
    for name in ("kv_num", "kv_idx", "full_kv_num", "full_kv_idx", "block_class", "q_num", "q_idx", "full_q_num",
                 "full_q_idx"):
        assert np.array_equal(ts[name], td[name]), name
    q = workloads.bf16_torch(dec.q_bits, dev)
    kp = workloads.bf16_torch(dec.k_bits, dev)
    vp = workloads.bf16_torch(dec.v_bits, dev)
    pt = torch.from_numpy(dec.page_table).to(dev)
    out, lse = fa.flex_decode(q, kp, vp, pt, sel, None, dec.scale, status=status, out_dtype=torch.float32)
    assert fa.check_status(status) == fa.OK
    q64, k64, v64 = (synth.bf16_bits_to_f64(x) for x in (dec.q_bits, dec.k_bits, dec.v_bits))
    o_ref, lse_ref = orc.decode_attention(q64, k64, v64, dec.page_table, dec.kv_lens, dec.rule, dec.scale, None,
                                          doc_ids=ids if kind == "doc" else None, requests=list(range(dec.Bz)),
                                          kv_len_table=L)
    gc.compare(out.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, f"prebuilt {kind} page={page} bq={bq}")


def test_prebuilt_mask_position_out_of_range():
    dec = workloads.cfg5(Bz=3, Hq=4, Hkv=2, d=64, page=64, lo=1, hi=5 * 64)
    dec.generate()
    L = dec.kv_len
    big = fa.create_block_mask(fa.make_mask_rule(dec.rule), 1, dec.Hq, L, L, 128, 64)
    qpos = torch.tensor([5, L + 300, -2], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sel = fa.select_rows(big, qpos, status=status)
    assert fa.check_status(status) == fa.ERR_DEVICE_CHECK
    ts = gc.tables_np(sel)
    assert ts["kv_num"][1:, 0, 0].tolist() == [0, 0] and ts["full_kv_num"][1:, 0, 0].tolist() == [0, 0]
    # position 5 under causal: key block 0 partial (keys 0..5 of 0..63), nothing else
    assert ts["kv_num"][0, 0, 0] == 1 and ts["kv_idx"][0, 0, 0, 0] == 0 and ts["full_kv_num"][0, 0, 0] == 0
    assert not ts["block_class"][1:].any()
