"""fa_flex_forward_split (long rows cut into chunks of key blocks, each a tile with its own softmax state,
merged by the LSE-weighted law) on the GPU against the fp64 oracle on the same seeded inputs.

Small cases compare every element (ragged tails, chunks of 1, 2 and 3 blocks so that rows split into many
chunks and some chunks are empty, every rule kind and score kind, two-tile pairing by rows (MHA) and by
sibling heads (GQA), bf16 and fp32 output, empty rows); a long causal sequence is compared at full size
on sampled rows of every query block, and against the unsplit forward.
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
DOC = np.repeat(np.arange(7, dtype=np.int32), [40, 3, 100, 17, 60, 9, 200 + 600])[None, :]


def run_split(w, chunk, out_dtype=torch.float32, status=None):
    dev = "cuda"
    q = workloads.bf16_torch(w.q_bits, dev)
    k = workloads.bf16_torch(w.k_bits, dev)
    v = workloads.bf16_torch(w.v_bits, dev)
    doc = gc.rule_arrays(w, dev)
    rule = fa.make_mask_rule(w.rule, doc_ids=doc)
    bm = fa.create_block_mask(rule, w.B, w.Hq, w.q_len, w.kv_len, w.bq, w.bk, device=dev, keep=[doc])
    al, rb, sc = gc.score_tensors(w.score, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev) if status is None else status
    out, lse = fa.flex_forward_split(q, k, v, bm, sc, w.scale, chunk_blocks=chunk, status=st, out_dtype=out_dtype)
    assert fa.check_status(st) == fa.OK
    ref_out, ref_lse = fa.flex_forward(q, k, v, bm, sc, w.scale, status=st, out_dtype=out_dtype)
    assert fa.check_status(st) == fa.OK
    return out, lse, ref_out, ref_lse, (al, rb, doc)


CASES = [
    # name, B, Hq, Hkv, N, d, rule, score
    ("causal_ragged_mha", 2, 3, 3, 1000, 128, [("causal",)], {}),
    ("causal_gqa", 1, 4, 2, 777, 128, [("causal",)], {}),
    ("window_softcap", 1, 2, 2, 900, 128, CW(300), dict(softcap=30.0)),
    ("doc_alibi", 1, 4, 4, 1029, 128, [("causal",), ("doc",), ("and",)], dict(alibi_slopes=workloads.alibi_slopes(4))),
    ("prefix_or_d64", 1, 2, 1, 640, 64, [("causal",), ("prefix", 200), ("or",)], {}),
    ("relbias", 1, 2, 2, 300, 64, CW(150), None),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("chunk", [1, 2, 3])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_split_small_all_elements(case, chunk, out_dtype):
    name, B, Hq, Hkv, n, d, rule, score = case
    if score is None:
        rng = np.random.default_rng(5)
        score = dict(rel_bias=(rng.standard_normal((Hq, 2 * n - 1)) * 2).astype(np.float32))
    w = workloads.Prefill(name, B, Hq, Hkv, n, n, d, 128, 128, rule, score, 1.0 / math.sqrt(d), 31)
    if any(op[0] == "doc" for op in rule):
        w.doc_ids = DOC[:, :n]
    w.generate()
    out, lse, ref_out, ref_lse, _ = run_split(w, chunk, out_dtype)
    qf, kf, vf = (synth.bf16_bits_to_f64(x) for x in (w.q_bits, w.k_bits, w.v_bits))
    o_ref, lse_ref = orc.attention(qf, kf, vf, w.rule, w.scale, gc.oracle_score(w.score), doc_ids=w.doc_ids)
    gc.compare(out.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, f"{name} chunk={chunk}",
               out_bf16=out_dtype == torch.bfloat16)


def test_split_empty_rows():
    # a prefix of length 0 allows nothing: every chunk is empty, O = 0 and LSE = -inf everywhere
    w = workloads.Prefill("empty", 1, 2, 2, 300, 300, 128, 128, 128, [("prefix", 0)], {}, 1.0 / math.sqrt(128), 3)
    w.generate()
    out, lse, _, _, _ = run_split(w, 1)
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


def test_split_long_causal_full_size():
    # causal N = 16384, two heads: rows of up to 128 key blocks cut into chunks of 16; every query block
    # compared with the oracle on its first, last and one random row; and with the unsplit forward
    w = workloads.Prefill("long_causal", 1, 2, 2, 16384, 16384, 128, 128, 128, [("causal",)], {},
                          1.0 / math.sqrt(128), 41).generate()
    out, lse, ref_out, ref_lse, _ = run_split(w, 16)
    per_block = gc.sample_rows_every_block(w, seed=4)
    rows = np.concatenate([np.asarray(x, dtype=np.int64) for x in per_block])
    ridx = torch.from_numpy(rows).cuda()
    o_all = out[:, :, ridx].cpu().numpy()
    l_all = lse[:, :, ridx].cpu().numpy()
    for h in range(w.Hq):
        o_ref, lse_ref = gc.oracle_rows_per_block(w, 0, h, per_block)
        gc.compare(o_all[0, h], l_all[0, h], o_ref, lse_ref, f"long causal h={h}")
    # the split and the unsplit forward agree within the tolerance everywhere
    d = (out - ref_out).abs()
    assert d.max().item() <= gc.O_MAX and d.mean().item() <= gc.O_MEAN
    assert (lse - ref_lse).abs().max().item() <= gc.LSE_MAX


@pytest.mark.parametrize("chunk", [2, 7])
def test_split_chunked_prefill_with_query_offset(chunk):
    # 300 new tokens (a ragged last block) at the end of a 4000-token context: causal in global positions
    # (query offset 3700), every element against the oracle
    q_len, kv_len = 300, 4000
    w = workloads.Prefill("chunked", 1, 4, 2, q_len, kv_len, 128, 128, 128, [("causal",)], {},
                          1.0 / math.sqrt(128), 17).generate()
    dev = "cuda"
    q = workloads.bf16_torch(w.q_bits, dev)
    k = workloads.bf16_torch(w.k_bits, dev)
    v = workloads.bf16_torch(w.v_bits, dev)
    off = torch.tensor([kv_len - q_len], dtype=torch.int32, device=dev)
    bm = fa.create_block_mask(fa.make_mask_rule(w.rule, q_offset=off, batch_dependent=True), 1, 4, q_len, kv_len,
                              128, 128, device=dev, keep=[off])
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = fa.flex_forward_split(q, k, v, bm, None, w.scale, chunk_blocks=chunk, status=st,
                                     out_dtype=torch.float32)
    assert fa.check_status(st) == fa.OK
    qf, kf, vf = (synth.bf16_bits_to_f64(x) for x in (w.q_bits, w.k_bits, w.v_bits))
    o_ref, lse_ref = orc.attention(qf, kf, vf, w.rule, w.scale, None, q_offset=np.array([kv_len - q_len]))
    gc.compare(out.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, f"chunked prefill chunk={chunk}")


def test_split_rejects_bad_arguments():
    w = workloads.Prefill("args", 1, 2, 2, 256, 256, 128, 64, 64, [("causal",)], {}, 1.0 / math.sqrt(128), 3)
    w.generate()
    q = workloads.bf16_torch(w.q_bits, "cuda")
    bm = fa.create_block_mask(fa.make_mask_rule(w.rule), 1, 2, 256, 256, 64, 64)
    with pytest.raises(fa.FaError) as e:   # 64 x 64 blocks: the split runs the tcgen05 kernel only
        fa.flex_forward_split(q, q, q, bm, None, None, chunk_blocks=2)
    assert e.value.code == fa.ERR_UNSUPPORTED
    bm2 = fa.create_block_mask(fa.make_mask_rule(w.rule), 1, 2, 256, 256, 128, 128)
    with pytest.raises(fa.FaError) as e:
        fa.flex_forward_split(q, q, q, bm2, None, None, chunk_blocks=0)
    assert e.value.code in (fa.ERR_SHAPE, fa.ERR_INVALID_ARG)
