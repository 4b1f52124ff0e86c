"""The allocation-free RMSNorm backward (mtk_rmsnorm_bwd_noalloc) against the regular entry point.

Callers that cannot allocate device memory where they need the kernel (code under a memory
manager that owns the whole device, or paths where cudaMalloc's implicit synchronisation is
not allowed) use this variant; its scratch is a fixed array inside the library. This file
is collected last so that a run stopping at the first failure has already run every other
test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from host_memory_streamed_stream_gb300 import _build, _lib

    _build.build()
    return _lib.load()


def _inputs(seed, T, h):
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = (torch.randn(T, h, generator=g) * 2.0).cuda()
    dy = torch.randn(T, h, generator=g).cuda()
    dres = torch.randn(T, h, generator=g).cuda()
    gamma = (1.0 + 0.5 * torch.randn(h, generator=g)).to(torch.bfloat16).cuda()
    rstd = torch.rsqrt(x.pow(2).mean(dim=1) + 1e-5).float()
    return x, dy, dres, gamma, rstd


def _call(lib, noalloc, x, dy, dres, gamma, rstd):
    T, h = x.shape
    dx = torch.empty(T, h, device="cuda")
    dxb = torch.empty(T, h, dtype=torch.bfloat16, device="cuda")
    dg = torch.empty(h, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    if noalloc:
        rc = lib.mtk_rmsnorm_bwd_noalloc(dy.data_ptr(), x.data_ptr(), gamma.data_ptr(), rstd.data_ptr(),
                                         dres.data_ptr(), dx.data_ptr(), dxb.data_ptr(), dg.data_ptr(), T, h, s)
    else:
        partial = torch.empty(lib.mtk_rmsnorm_bwd_parts(T), h, device="cuda")
        rc = lib.mtk_rmsnorm_bwd(dy.data_ptr(), x.data_ptr(), gamma.data_ptr(), rstd.data_ptr(), dres.data_ptr(),
                                 dx.data_ptr(), dxb.data_ptr(), partial.data_ptr(), dg.data_ptr(), T, h, s)
    assert rc == 0, (noalloc, rc, lib.mt_last_error(None))
    torch.cuda.synchronize()
    return dx, dxb, dg


def _close(a, b, tol):
    a, b = a.float(), b.float()
    return (a - b).abs().max().item() <= tol * max(b.abs().max().item(), 1e-30)


def test_noalloc_matches_regular_entry_point_twice(lib):
    # two calls in a row, different sizes and data: the shared scratch keeps the first call's
    # contents, which must not leak into the second
    for seed, (T, h) in ((1, (1000, 4096)), (2, (37, 5120))):
        inp = _inputs(seed, T, h)
        ref = _call(lib, False, *inp)
        got = _call(lib, True, *inp)
        assert _close(got[0], ref[0], 1e-5)   # fp32 dx, as in the kernel tests
        assert _close(got[1], ref[1], 4e-3)   # bf16 copy of dx
        assert _close(got[2], ref[2], 4e-3)   # bf16 dgamma


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    T, h = 304, 8200  # min(T, 304) * h > 304 * 8192
    x = torch.zeros(1, device="cuda")
    rc = lib.mtk_rmsnorm_bwd_noalloc(x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), None, x.data_ptr(),
                                     None, x.data_ptr(), T, h, None)
    assert rc == -1
    assert b"exceeds the fixed scratch" in lib.mt_last_error(None)
