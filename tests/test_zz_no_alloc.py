"""The allocation-free decode entry point (fa_flex_decode_noalloc).

It serves callers that cannot pass a device workspace: programs whose device memory is owned by another
runtime's pool, and serving loops that must never call cudaMalloc / cudaFree (cudaFree synchronises the
device). It must give the same results as fa_flex_decode, call after call, using only the library's fixed
device array; a problem too large for that array must be refused before anything runs.

This file is named to be collected last, so a run that stops at the first failure has run every other
test before it. It passes alone in a fresh process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

from block_sparse_masked_create_gb300 import fa, workloads

pytestmark = pytest.mark.gpu


def _setup(dec):
    dev = "cuda"
    q = workloads.bf16_torch(dec.q_bits, dev)
    kp = workloads.bf16_torch(dec.k_bits, dev)
    vp = workloads.bf16_torch(dec.v_bits, dev)
    pt = torch.from_numpy(np.ascontiguousarray(dec.page_table)).to(dev)
    off = torch.from_numpy(dec.q_offset).to(dev)
    rule = fa.make_mask_rule(dec.rule, q_offset=off, batch_dependent=True)
    bm = fa.create_block_mask(rule, dec.Bz, dec.Hq, 1, dec.kv_len, 1, dec.page, keep=[off])
    return q, kp, vp, pt, bm


def _same_bits(x: torch.Tensor, y: torch.Tensor) -> bool:
    iv = torch.int16 if x.dtype == torch.bfloat16 else torch.int32
    return torch.equal(x.contiguous().view(iv).cpu(), y.contiguous().view(iv).cpu())


def _both(dec, out_dtype, status):
    """fa_flex_decode (caller workspace) and fa_flex_decode_noalloc (the library's array) on the same
    inputs; the no-alloc outputs start as NaN so that anything it leaves unwritten shows."""
    q, kp, vp, pt, bm = _setup(dec)
    ref_o, ref_l = fa.flex_decode(q, kp, vp, pt, bm, None, dec.scale, status=status, out_dtype=out_dtype)
    assert fa.check_status(status) == fa.OK
    out = torch.full(q.shape, float("nan"), dtype=out_dtype, device="cuda")
    lse = torch.full((dec.Bz, dec.Hq), float("nan"), dtype=torch.float32, device="cuda")
    code = fa.flex_decode_noalloc(q, kp, vp, pt, bm, None, dec.scale, out=out, lse=lse, status=status)
    assert code == fa.OK, fa.status_string(code)
    assert fa.check_status(status) == fa.OK
    return out, lse, ref_o, ref_l


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_noalloc_decode_matches_workspace_decode_twice(out_dtype):
    # Two calls on the full 64-request workload with a call on other inputs between them: a smaller batch
    # with other lengths and a shorter table, so the split slots of the shared array hold different data when
    # the second full call starts. Every call must equal fa_flex_decode on the same inputs bit for bit:
    # both run the same kernels on the same inputs, and only the workspace differs.
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    full = workloads.cfg5().generate()
    need = fa.decode_workspace_bytes(full.Bz, full.Hq, full.d, full.max_pages, full.page)
    assert 0 < need <= fa.decode_noalloc_scratch_bytes()
    other = workloads.cfg5(Bz=9, lo=3000, hi=20000).generate()
    for call, dec in enumerate((full, other, full)):
        out, lse, ref_o, ref_l = _both(dec, out_dtype, status)
        assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all(), f"call {call}"
        assert _same_bits(out, ref_o), f"call {call}: O differs from fa_flex_decode"
        assert _same_bits(lse, ref_l), f"call {call}: LSE differs from fa_flex_decode"


def test_noalloc_decode_refuses_oversized_problems():
    # A problem whose split workspace exceeds the fixed array, with every other argument valid: a table
    # shared by all requests (no per-request state, Bm = 1) declared for a batch far larger than the array
    # can hold. fa_flex_decode checks all other arguments first, so the refusal is the size, and nothing is
    # launched (the batch is never touched).
    dec = workloads.cfg5(Bz=2, Hq=4, Hkv=2, d=64, page=32, lo=40, hi=200).generate()
    q, kp, vp, pt, _ = _setup(dec)
    shared = fa.create_block_mask(fa.make_mask_rule([("causal",)]), 1, dec.Hq, 1, dec.kv_len, 1, dec.page)
    big_bz = 1 << 17
    assert fa.decode_workspace_bytes(big_bz, dec.Hq, dec.d, dec.max_pages, dec.page) > \
        fa.decode_noalloc_scratch_bytes()
    lib = fa.load()
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    lse = torch.empty((dec.Bz, dec.Hq), dtype=torch.float32, device="cuda")

    def call(bz, d):
        return lib.fa_flex_decode_noalloc(fa._ptr(q), fa._ptr(kp), fa._ptr(vp), fa._ptr(pt), kp.shape[0],
                                          fa.ctypes.byref(shared.c), None, 0.0, fa._ptr(out), 1, fa._ptr(lse), bz,
                                          dec.Hq, dec.Hkv, d, dec.page, dec.max_pages, None, None,
                                          fa._stream(q.device))

    assert call(big_bz, dec.d) == fa.ERR_BUFFER
    # another argument error in the same call keeps the code fa_flex_decode gives it
    assert call(big_bz, 96) == fa.ERR_UNSUPPORTED
    torch.cuda.synchronize()
