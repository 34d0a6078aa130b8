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
from tests import gpu_common as gc

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


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_noalloc_decode_matches_workspace_decode_twice(out_dtype):
    dec = workloads.cfg5().generate()          # the full 64-request workload fits the fixed array
    need = fa.decode_workspace_bytes(dec.Bz, dec.Hq, dec.d, dec.max_pages, dec.page)
    assert 0 < need <= fa.decode_noalloc_scratch_bytes()
    q, kp, vp, pt, bm = _setup(dec)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref_o, ref_l = fa.flex_decode(q, kp, vp, pt, bm, None, dec.scale, status=status, out_dtype=out_dtype)
    assert fa.check_status(status) == fa.OK
    for call in range(2):                      # the shared array keeps the previous call's contents
        out = torch.full(q.shape, float("nan"), dtype=out_dtype, device="cuda")
        lse = torch.full((dec.Bz, dec.Hq), float("nan"), dtype=torch.float32, device="cuda")
        code = fa.flex_decode_noalloc(q, kp, vp, pt, bm, None, dec.scale, out=out, lse=lse, status=status)
        assert code == fa.OK, fa.status_string(code)
        assert fa.check_status(status) == fa.OK
        o, l, ro, rl = (x.float().cpu().numpy() for x in (out, lse, ref_o, ref_l))
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))
        err = np.abs(o - ro)
        assert err.max() <= gc.O_MAX and err.mean() <= gc.O_MEAN, f"call {call}: max {err.max():.3e}"
        assert np.abs(l - rl).max() <= gc.LSE_MAX, f"call {call}"


def test_noalloc_decode_refuses_oversized_problems():
    dec = workloads.cfg5(Bz=2, Hq=4, Hkv=2, d=64, page=32, lo=40, hi=200).generate()
    q, kp, vp, pt, bm = _setup(dec)
    # same pages and table, but declared for a batch far larger than the fixed array can hold
    big_bz = 1 << 17
    assert fa.decode_workspace_bytes(big_bz, dec.Hq, dec.d, dec.max_pages, dec.page) > \
        fa.decode_noalloc_scratch_bytes()
    lib = fa.load()
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    lse = torch.empty((dec.Bz, dec.Hq), dtype=torch.float32, device="cuda")
    code = lib.fa_flex_decode_noalloc(fa._ptr(q), fa._ptr(kp), fa._ptr(vp), fa._ptr(pt), kp.shape[0],
                                      fa.ctypes.byref(bm.c), None, 0.0, fa._ptr(out), 1, fa._ptr(lse), big_bz,
                                      dec.Hq, dec.Hkv, dec.d, dec.page, dec.max_pages, None, None,
                                      fa._stream(q.device))
    assert code == fa.ERR_BUFFER
