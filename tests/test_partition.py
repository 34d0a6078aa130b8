"""Partition of a prefill across ranks by (batch row, KV head) units, on CPU: every unit is owned by exactly
one rank, ranges are balanced, two gloo ranks agree on that, and the ranks' outputs (the fp64 oracle run on
each rank's local problems, with the per-head and per-batch state sliced to match) concatenate to the
oracle's output for the whole problem."""
import math
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from block_sparse_masked_create_gb300 import partition, synth, workloads
from oracle import flexmask_oracle as orc


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("B,Hkv,world", [(4, 16, 1), (4, 16, 2), (4, 16, 3), (8, 16, 8), (1, 8, 16), (3, 5, 4),
                                         (2, 1, 3), (7, 3, 5)])
def test_pieces_cover_every_unit_once(B, Hkv, world):
    seen = []
    sizes = []
    for r in range(world):
        pieces = partition.pieces_for_rank(B, Hkv, world, r)
        assert len(pieces) <= 3
        for (b0, b1, h0, h1) in pieces:
            assert 0 <= b0 < b1 <= B and 0 <= h0 < h1 <= Hkv
        u = partition.units_of(pieces)
        sizes.append(len(u))
        seen += u
    assert sorted(seen) == sorted((b, h) for b in range(B) for h in range(Hkv))
    assert max(sizes) - min(sizes) <= 1


def _tiny():
    B, Hq, Hkv, n, d = 3, 6, 3, 96, 32
    w = workloads.Prefill("tiny_gqa_doc_alibi", B, Hq, Hkv, n, n, d, 16, 16, [("causal",), ("doc",), ("and",)],
                          dict(alibi_slopes=workloads.alibi_slopes(Hq)), 1.0 / math.sqrt(d), 99).generate()
    rng = np.random.default_rng(2)
    w.doc_ids = np.sort(rng.integers(0, 4, size=(B, n)), axis=1).astype(np.int32)
    off = np.array([0, 5, 11], dtype=np.int32)
    return w, off


def _oracle(w, off):
    qf, kf, vf = (synth.bf16_bits_to_f64(x) for x in (w.q_bits, w.k_bits, w.v_bits))
    sc = {"alibi_slopes": np.asarray(w.score["alibi_slopes"], np.float32).astype(np.float64)}
    return orc.attention(qf, kf, vf, w.rule, w.scale, sc, q_offset=off, doc_ids=w.doc_ids)


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, off = _tiny()
        pieces = partition.pieces_for_rank(w.B, w.Hkv, world, rank)
        results = []
        for piece in pieces:
            loc, loff = partition.slice_prefill(w, piece, off)
            o, l = _oracle(loc, loff)
            results.append((piece, o, l))
        gathered = [None] * world
        dist.all_gather_object(gathered, (rank, partition.units_of(pieces), results))
        if rank == 0:
            out["gathered"] = gathered
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_concatenate_to_the_whole_problem():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    w, off = _tiny()
    units = [u for (_, us, _) in out["gathered"] for u in us]
    assert sorted(units) == sorted((b, h) for b in range(w.B) for h in range(w.Hkv))   # exactly once
    g = w.Hq // w.Hkv
    o_all = np.full((w.B, w.Hq, w.q_len, w.d), np.nan)
    l_all = np.full((w.B, w.Hq, w.q_len), np.nan)
    for (_, _, results) in out["gathered"]:
        for (b0, b1, h0, h1), o, l in results:
            o_all[b0:b1, h0 * g:h1 * g] = o
            l_all[b0:b1, h0 * g:h1 * g] = l
    o_ref, l_ref = _oracle(w, off)
    assert np.array_equal(o_all, o_ref)
    assert np.array_equal(l_all, l_ref)


def test_slices_drawn_from_the_generator_equal_slices_of_the_whole():
    w, off = _tiny()
    bare = workloads.Prefill(w.name, w.B, w.Hq, w.Hkv, w.q_len, w.kv_len, w.d, w.bq, w.bk, w.rule, dict(w.score),
                             w.scale, w.seed)
    bare.doc_ids = w.doc_ids
    for piece in partition.pieces_for_rank(w.B, w.Hkv, 4, 1) + partition.pieces_for_rank(w.B, w.Hkv, 4, 3):
        a, _ = partition.slice_prefill(w, piece, off)
        b, _ = partition.slice_prefill(bare, piece, off)
        assert np.array_equal(a.q_bits, b.q_bits) and np.array_equal(a.k_bits, b.k_bits)
        assert np.array_equal(a.v_bits, b.v_bits)
