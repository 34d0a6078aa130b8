"""The partition by (batch row, KV head) units with real kernels: every rank's local problems (sliced inputs,
sliced ALiBi slopes and document ids, a mask rebuilt per piece) run through the C ABI on one GPU, and their
outputs put together equal the forward of the whole problem bit for bit (a row's result does not depend on
which other rows share its launch)."""
import math

import numpy as np
import pytest
import torch

from block_sparse_masked_create_gb300 import fa, partition, workloads
from tests import gpu_common as gc

pytestmark = pytest.mark.gpu


def _forward(w, off):
    dev = "cuda"
    q = workloads.bf16_torch(w.q_bits, dev)
    k = workloads.bf16_torch(w.k_bits, dev)
    v = workloads.bf16_torch(w.v_bits, dev)
    doc = gc.rule_arrays(w, dev)
    off_t = None if off is None else torch.from_numpy(np.ascontiguousarray(off.astype(np.int32))).to(dev)
    rule = fa.make_mask_rule(w.rule, doc_ids=doc, q_offset=off_t, batch_dependent=True)
    bm = fa.create_block_mask(rule, w.B, w.Hq, w.q_len, w.kv_len, w.bq, w.bk, device=dev, keep=[doc, off_t])
    al, rb, sc = gc.score_tensors(w.score, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = fa.flex_forward(q, k, v, bm, sc, w.scale, status=st, out_dtype=torch.float32)
    assert fa.check_status(st) == fa.OK
    return out.cpu(), lse.cpu()


@pytest.mark.parametrize("world", [2, 3, 5])
def test_pieces_of_all_ranks_reproduce_the_whole_forward(world):
    B, Hq, Hkv, n = 3, 8, 4, 640
    w = workloads.Prefill("part_gqa_doc_alibi", B, Hq, Hkv, n, n, 128, 128, 128, [("causal",), ("doc",), ("and",)],
                          dict(alibi_slopes=workloads.alibi_slopes(Hq)), 1.0 / math.sqrt(128), 123).generate()
    rng = np.random.default_rng(9)
    w.doc_ids = np.sort(rng.integers(0, 3, size=(B, n)), axis=1).astype(np.int32)
    off = np.array([0, 64, 200], dtype=np.int32)
    o_ref, l_ref = _forward(w, off)
    g = Hq // Hkv
    o_all = torch.full_like(o_ref, float("nan"))
    l_all = torch.full_like(l_ref, float("nan"))
    for r in range(world):
        for piece in partition.pieces_for_rank(B, Hkv, world, r):
            loc, loff = partition.slice_prefill(w, piece, off)
            o, l = _forward(loc, loff)
            b0, b1, h0, h1 = piece
            o_all[b0:b1, h0 * g:h1 * g] = o
            l_all[b0:b1, h0 * g:h1 * g] = l
    assert torch.equal(o_all.view(torch.int32), o_ref.view(torch.int32))
    assert torch.equal(l_all.view(torch.int32), l_ref.view(torch.int32))
