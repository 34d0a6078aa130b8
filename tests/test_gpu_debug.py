"""GPU self-tests of the building blocks: the bounded pipeline wait, and the tcgen05 descriptor encodings
(one 128x128xK MMA chain vs a library GEMM on the same bf16 inputs)."""
import pytest
import torch

from block_sparse_masked_create_gb300 import fa

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert fa.debug_wait_timeout(status, 2_000_000) == fa.OK     # 2 ms limit, nothing ever arrives
    assert fa.check_status(status) == fa.ERR_TIMEOUT
    # the context is still usable afterwards
    x = torch.arange(10, device="cuda").sum().item()
    assert x == 45


@pytest.mark.parametrize("c", [20.0, 50.0])
def test_softcap_error_bound(c):
    # the kernels' soft-cap against fp64 c * tanh(x / c), over scores far beyond the cap
    x = torch.cat([torch.linspace(-8 * c, 8 * c, 1 << 20, dtype=torch.float64),
                   torch.randn(1 << 16, dtype=torch.float64) * 4.0]).float().cuda()
    y = fa.debug_softcap(x, c)
    ref = c * torch.tanh(x.double() / c)
    err = (y.double() - ref).abs()
    assert err.max().item() < c * 2e-5, err.max().item()
    small = x.abs() < c / 2
    rel = (err[small] / ref[small].abs().clamp_min(1e-30)).max().item()
    assert rel < 3e-5, rel
    assert bool((y.abs() <= c).all())


@pytest.mark.parametrize("K", [64, 128])
@pytest.mark.parametrize("b_mn", [False, True])
@pytest.mark.parametrize("use_tma", [0, 1, 2], ids=["st", "tma", "a_tmem"])
def test_tc5_gemm_descriptors(K, b_mn, use_tma):
    g = torch.Generator(device="cpu").manual_seed(K * 4 + 2 * b_mn + use_tma)
    A = torch.randn(128, K, generator=g).to(torch.bfloat16).cuda()
    B = (torch.randn(K, 128, generator=g) if b_mn else torch.randn(128, K, generator=g)).to(torch.bfloat16).cuda()
    C = torch.full((128, 128), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert fa.debug_tc5_gemm(A, B, C, K, b_mn, use_tma, status) == fa.OK
    assert fa.check_status(status) == fa.OK
    ref = A.double() @ (B.double() if b_mn else B.double().T)
    err = (C.double() - ref).abs().max().item()
    assert err < 1e-3, f"tcgen05 GEMM K={K} b_mn={b_mn} tma={use_tma}: max err {err}"
