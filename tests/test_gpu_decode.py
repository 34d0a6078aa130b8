"""fa_flex_decode (paged split-KV) on the GPU vs the fp64 paged oracle on the same seeded inputs: small
cases on every element, the 64-request workload at full size on a seeded sample of requests, and the
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


def test_cfg5_full_size_sampled():
    dec = workloads.cfg5().generate()
    out, lse, st, cnt = run_decode(dec)
    assert st == fa.OK
    L = dec.kv_lens
    reqs = sorted({int(np.argmin(L)), int(np.argmax(L))} | set(np.random.default_rng(2).integers(0, 64, 10).tolist()))
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
