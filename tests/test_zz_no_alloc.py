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


def test_noalloc_matches_regular_entry_point_twice(lib):
    # two calls in a row, different sizes and data: the shared scratch keeps the first call's
    # contents, which must not leak into the second. Both entry points run the same kernels
    # with the same fixed reduction order, so the outputs are bit-identical.
    for seed, (T, h) in ((1, (1000, 4096)), (2, (37, 5120))):
        inp = _inputs(seed, T, h)
        ref = _call(lib, False, *inp)
        got = _call(lib, True, *inp)
        for a, b in zip(got, ref):
            assert torch.equal(a, b)


def test_noalloc_calls_allocate_no_device_memory(lib):
    T, h = 640, 2048
    inp = _inputs(3, T, h)
    outs = [torch.empty(T, h, device="cuda"), torch.empty(T, h, dtype=torch.bfloat16, device="cuda"),
            torch.empty(h, dtype=torch.bfloat16, device="cuda")]
    x, dy, dres, gamma, rstd = inp
    s = torch.cuda.current_stream().cuda_stream

    def call():
        rc = lib.mtk_rmsnorm_bwd_noalloc(dy.data_ptr(), x.data_ptr(), gamma.data_ptr(), rstd.data_ptr(),
                                         dres.data_ptr(), outs[0].data_ptr(), outs[1].data_ptr(),
                                         outs[2].data_ptr(), T, h, s)
        assert rc == 0, lib.mt_last_error(None)

    call()  # the first call on a device may load the module that holds the fixed scratch
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0


def test_noalloc_rejects_misaligned_rows(lib):
    # a row slice starting one float in: the float4 accesses would fault, so nothing is launched
    T, h = 64, 1024
    x, dy, dres, gamma, rstd = _inputs(4, T + 1, h)
    dx = torch.empty(T + 1, h, device="cuda")
    dg = torch.empty(h, dtype=torch.bfloat16, device="cuda")
    off = 4  # bytes
    rc = lib.mtk_rmsnorm_bwd_noalloc(dy.data_ptr() + off, x.data_ptr(), gamma.data_ptr(), rstd.data_ptr(), None,
                                     dx.data_ptr(), None, dg.data_ptr(), T, h, None)
    assert rc == -1
    assert b"aligned" in lib.mt_last_error(None)
    torch.cuda.synchronize()  # the context is unharmed


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    T, h = 304, 8200  # min(T, 304) * h > 304 * 8192
    x = torch.zeros(1, device="cuda")
    rc = lib.mtk_rmsnorm_bwd_noalloc(x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), None, x.data_ptr(),
                                     None, x.data_ptr(), T, h, None)
    assert rc == -1
    assert b"exceeds the fixed scratch" in lib.mt_last_error(None)
