"""fa_flex_forward_paged on the GPU: K/V in a paged cache, one page per key block, pages in a seeded
shuffled order. The rules stay in logical positions, so the result must equal the contiguous forward
bit for bit (same kernel, same arithmetic, only the fetch addresses differ) and the fp64 oracle within
the forward tolerance. Covers the tcgen05 kernel (128-token pages) and the mma.sync kernel (64-token
pages), chunked prefill with per-request query offsets over a cached prefix, pages shared by two
requests, slots past the sequence holding junk, and a bad page id reported as a device-check error."""
import math

import numpy as np
import pytest
import torch

from block_sparse_masked_create_gb300 import fa, synth, workloads
from oracle import flexmask_oracle as orc
from tests import gpu_common as gc

pytestmark = pytest.mark.gpu

JUNK = 1.0e4  # finite value in page slots past the sequence: masked, so it must not show up


def to_pages(bits: np.ndarray, lens, page: int, seed: int, spare: int = 3):
    """bf16 bits [B, Hkv, N, d] -> pages [P, Hkv, page, d] (bits) and table [B, max_pages] int32. Request b
    keeps ceil(lens[b] / page) pages, placed at shuffled physical ids; slots past lens[b] hold JUNK and
    the table's unused entries are -1."""
    B, Hkv, N, d = bits.shape
    max_pages = -(-N // page)
    need = [-(-int(L) // page) for L in lens]
    P = sum(need) + spare
    perm = np.random.default_rng(seed).permutation(P).astype(np.int32)
    junk = synth.bf16_bits_from_double(JUNK)
    pages = np.full((P, Hkv, page, d), junk, dtype=np.uint16)
    table = np.full((B, max_pages), -1, dtype=np.int32)
    nxt = 0
    for b in range(B):
        for c in range(need[b]):
            pid = int(perm[nxt])
            nxt += 1
            table[b, c] = pid
            j0, j1 = c * page, min((c + 1) * page, int(lens[b]))
            pages[pid, :, : j1 - j0] = bits[b, :, j0:j1]
    return pages, table


def run_paged(w, k_pages, v_pages, table, q_off=None, out_dtype=torch.float32, bq=None, bk=None):
    dev = "cuda"
    q = workloads.bf16_torch(w.q_bits, dev)
    kp = workloads.bf16_torch(k_pages, dev)
    vp = workloads.bf16_torch(v_pages, dev)
    pt = torch.from_numpy(table).to(dev)
    off = None if q_off is None else torch.from_numpy(np.asarray(q_off, np.int32)).to(dev)
    doc = gc.rule_arrays(w, dev)
    rule = fa.make_mask_rule(w.rule, doc_ids=doc, q_offset=off)
    bm = fa.create_block_mask(rule, w.B, w.Hq, w.q_len, w.kv_len, bq or w.bq, bk or w.bk, device=dev,
                              keep=[doc, off])
    al, rb, sc = gc.score_tensors(w.score, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = fa.flex_forward_paged(q, kp, vp, pt, bm, w.kv_len, sc, w.scale, status=status, out_dtype=out_dtype)
    st = fa.check_status(status)
    return out.cpu().numpy(), lse.cpu().numpy(), st, (al, rb, doc, off, q, kp, vp, pt, bm)


def prefill(name, B, Hq, Hkv, q_len, kv_len, d, bq, bk, rule, score=None, seed=31):
    w = workloads.Prefill(name, B, Hq, Hkv, q_len, kv_len, d, bq, bk, rule, score or {}, 1.0 / math.sqrt(d), seed)
    return w.generate()


CASES = [
    # (name, B, Hq, Hkv, N, d, block, rule, score)
    ("causal_gqa_tc5", 2, 4, 2, 700, 128, 128, [("causal",)], None),
    ("window_softcap_tc5_d64", 1, 2, 2, 1000, 64, 128, [("causal",), ("window", 300), ("and",)], {"softcap": 20.0}),
    ("prefix_or_causal_mma", 2, 2, 1, 333, 128, 64, [("causal",), ("prefix", 70), ("or",)], None),
    ("dense_alibi_mma_d64", 1, 4, 4, 200, 64, 64, [("true",)], {"alibi_slopes": [0.5, 0.25, 0.125, 0.0625]}),
]


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_paged_equals_contiguous_and_oracle(ci):
    name, B, Hq, Hkv, N, d, blk, rule, score = CASES[ci]
    w = prefill(name, B, Hq, Hkv, N, N, d, blk, blk, rule, score)
    lens = [N] * B
    kp, table = to_pages(w.k_bits, lens, blk, seed=100 + ci)
    vp, _ = to_pages(w.v_bits, lens, blk, seed=100 + ci)
    o_p, lse_p, st, _keep = run_paged(w, kp, vp, table)
    assert st == fa.OK
    r = gc.run_prefill(w, out_dtype=torch.float32)
    assert r["status"] == fa.OK
    o_c, lse_c = r["out"].cpu().numpy(), r["lse"].cpu().numpy()
    assert np.array_equal(o_p.view(np.uint32), o_c.view(np.uint32)), "paged O differs from the contiguous O"
    assert np.array_equal(lse_p.view(np.uint32), lse_c.view(np.uint32)), "paged LSE differs"
    o_ref, lse_ref = orc.attention(synth.bf16_bits_to_f64(w.q_bits), synth.bf16_bits_to_f64(w.k_bits),
                                   synth.bf16_bits_to_f64(w.v_bits), w.rule, w.scale, gc.oracle_score(w.score))
    gc.compare(o_p, lse_p, o_ref, lse_ref, name)


@pytest.mark.parametrize("blk", [128, 64])
def test_chunked_prefill_over_a_cached_prefix(blk):
    # two requests add 200 new tokens each after cached prefixes of 300 and 900 tokens: the query at
    # local row i sits at global position prefix_b + i, and the causal rule then also stops every row
    # at its request's own length; keys past it sit in junk-filled slots or unlisted pages
    B, Hq, Hkv, d, q_len = 2, 4, 1, 128, 200
    prefix = np.array([300, 900], np.int32)
    lens = prefix + q_len
    kv_len = int(lens.max())
    w = prefill(f"chunked_{blk}", B, Hq, Hkv, q_len, kv_len, d, blk, blk, [("causal",)], seed=41)
    kp, table = to_pages(w.k_bits, lens, blk, seed=7)
    vp, _ = to_pages(w.v_bits, lens, blk, seed=7)
    o_p, lse_p, st, _keep = run_paged(w, kp, vp, table, q_off=prefix)
    assert st == fa.OK
    o_ref, lse_ref = orc.attention(synth.bf16_bits_to_f64(w.q_bits), synth.bf16_bits_to_f64(w.k_bits),
                                   synth.bf16_bits_to_f64(w.v_bits), w.rule, w.scale, None, q_offset=prefix)
    gc.compare(o_p, lse_p, o_ref, lse_ref, f"chunked_{blk}")


def test_shared_prefix_pages():
    # request 1 reuses request 0's physical pages for the first 3 blocks (a shared prompt prefix); its
    # logical K/V there are request 0's, which the contiguous reference copies in
    B, Hq, Hkv, d, N, blk = 2, 2, 2, 128, 640, 128
    w = prefill("shared_prefix", B, Hq, Hkv, N, N, d, blk, blk, [("causal",)], seed=51)
    shared = 3 * blk
    w.k_bits[1, :, :shared] = w.k_bits[0, :, :shared]
    w.v_bits[1, :, :shared] = w.v_bits[0, :, :shared]
    kp, table = to_pages(w.k_bits, [N, N], blk, seed=9)
    vp, _ = to_pages(w.v_bits, [N, N], blk, seed=9)
    table[1, :3] = table[0, :3]  # request 1's own copies of those pages are left unused
    o_p, lse_p, st, _keep = run_paged(w, kp, vp, table)
    assert st == fa.OK
    r = gc.run_prefill(w, out_dtype=torch.float32)
    assert np.array_equal(o_p.view(np.uint32), r["out"].cpu().numpy().view(np.uint32))
    assert np.array_equal(lse_p.view(np.uint32), r["lse"].cpu().numpy().view(np.uint32))


@pytest.mark.parametrize("blk", [128, 64])
def test_bad_page_id_is_reported(blk):
    # a listed block names a page id past the pool: the kernel reads page 0 instead (in bounds) and sets
    # the device-check status; the context stays usable
    B, Hq, Hkv, d, N = 1, 2, 2, 128, 4 * blk
    w = prefill("bad_page", B, Hq, Hkv, N, N, d, blk, blk, [("causal",)], seed=61)
    kp, table = to_pages(w.k_bits, [N], blk, seed=3)
    vp, _ = to_pages(w.v_bits, [N], blk, seed=3)
    table[0, 2] = kp.shape[0] + 5
    _, _, st, _keep = run_paged(w, kp, vp, table)
    assert st == fa.ERR_DEVICE_CHECK
    table[0, 2] = -1
    _, _, st2, _keep2 = run_paged(w, kp, vp, table)
    assert st2 == fa.ERR_DEVICE_CHECK
    r = gc.run_prefill(w)  # the next call on the same context runs normally
    assert r["status"] == fa.OK


def test_page_size_must_match_the_key_block():
    w = prefill("page_mismatch", 1, 2, 2, 256, 256, 128, 128, 128, [("causal",)], seed=71)
    kp, table = to_pages(w.k_bits, [256], 64, seed=1)
    vp, _ = to_pages(w.v_bits, [256], 64, seed=1)
    with pytest.raises(fa.FaError) as e:
        run_paged(w, kp, vp, table)
    assert e.value.code == fa.ERR_SHAPE


def test_paged_cfg2_full_size_equals_contiguous():
    # the benchmarked configuration with K/V in 128-token pages at shuffled ids (the bench's paged line):
    # bit-identical to the contiguous forward
    w = workloads.cfg2().generate()
    kpb, table = workloads.paged_kv(w.k_bits, 128, w.seed)
    vpb, _ = workloads.paged_kv(w.v_bits, 128, w.seed)
    o_p, lse_p, st, _keep = run_paged(w, kpb, vpb, table)
    assert st == fa.OK
    r = gc.run_prefill(w, out_dtype=torch.float32)
    assert np.array_equal(o_p.view(np.uint32), r["out"].cpu().numpy().view(np.uint32))
    assert np.array_equal(lse_p.view(np.uint32), r["lse"].cpu().numpy().view(np.uint32))
