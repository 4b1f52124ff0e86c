"""The GEMM with its last, partial wave split over K (a split workspace set), against the
oracle's products and against the same GEMM without the split.

The split only reorders the K sum of the last wave's tiles: fp32 results stay within
fp32-accumulation error of the float64 oracle, bf16 results within the kernel tests' bars,
repeated launches are bit-identical, and a shape whose tile count leaves no partial wave (or
too few k-blocks) gives the unsplit result bit for bit.
"""
import numpy as np
import pytest

import oracle
from oracle import model as om

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    from host_memory_streamed_stream_gb300 import _build

    _build.build()
    from host_memory_streamed_stream_gb300 import kernels

    return kernels


@pytest.fixture
def split(K):
    """Run the test body with the split workspace set; turn the split off afterwards."""
    ws = K.gemm_use_workspace("cuda")
    yield ws
    K.gemm_use_workspace(None)
    torch.cuda.synchronize()


def _bf16(rng, shape, scale=1.0):
    x = oracle.bf16_bits_to_float(oracle.float_to_bf16_bits(rng.standard_normal(shape) * scale))
    return x, torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).cuda()


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


def _nerr(got, ref):
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))


def _splits(M, N, K_, paired=False):
    """Whether the library splits this shape (its rule, restated: the SM count, 128 x 256 tiles,
    128 x 128 output columns per tile when gate and up rows are paired, 64-wide k-blocks, at
    least 128 k-blocks and a last wave at most half full)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    g = min(sms, 256)
    bn = 128 if paired else 256
    tiles = -(-M // 128) * -(-N // bn)
    rem, kb = tiles % g, -(-K_ // 64)
    return rem != 0 and 2 * rem <= g and kb >= 128


# (M, N, K) of the forward product: fewer tiles than SMs with ragged edges and a ragged K, a
# small last wave after full waves, a last wave of 50 tiles, a last wave of 56 tiles, and a
# short K. The data and weight gradients of the same operands (K = N and K = M) are mostly
# below the split's k-block minimum and run unsplit, the 8192-token weight gradient splits.
SHAPES = [(1000, 776, 8200), (4096, 5120, 8192), (640, 2560, 8192), (8192, 2048, 8192), (300, 200, 256)]


@pytest.mark.parametrize("M,N,K_", SHAPES)
def test_split_gemm_layouts(K, split, M, N, K_):
    from host_memory_streamed_stream_gb300 import _lib

    lib = _lib.load()
    rng = np.random.default_rng(M * 7 + N + K_)
    x, xt = _bf16(rng, (M, K_))
    w, wt = _bf16(rng, (N, K_))
    dy, dyt = _bf16(rng, (M, N))
    cases = [  # forward, dgrad, wgrad: (A, a_mn, B, b_mn, M, N, K, reference)
        (xt, 0, wt, 0, M, N, K_, x @ w.T),
        (dyt, 0, wt, 1, M, K_, N, dy @ w),
        (dyt, 1, xt, 1, N, K_, M, dy.T @ x),
    ]
    for A, a_mn, B, b_mn, m, n, k, ref in cases:
        # fp32 accumulation over k random-sign terms: the kernel tests' 1e-5 bar (k <= 1024),
        # grown like sqrt(k)
        tol = 1e-5 * max(1.0, (k / 1024) ** 0.5)
        got = K.gemm(A, a_mn, B, b_mn, m, n, k, epi=K.EPI_STORE_F32)
        again = K.gemm(A, a_mn, B, b_mn, m, n, k, epi=K.EPI_STORE_F32)
        assert torch.equal(got, again)  # deterministic
        assert _nerr(_np(got), ref) < tol
        gb = K.gemm(A, a_mn, B, b_mn, m, n, k, epi=K.EPI_STORE_BF16)
        assert _nerr(_np(gb), ref) < 4e-3
        lib.mtk_gemm_use_workspace(None)
        plain = K.gemm(A, a_mn, B, b_mn, m, n, k, epi=K.EPI_STORE_F32)
        assert lib.mtk_gemm_use_workspace(split.data_ptr()) == 0
        if _splits(m, n, k):
            assert not torch.equal(got, plain)  # the K sum was reordered somewhere
        else:
            assert torch.equal(got, plain)
        assert _nerr(_np(got), _np(plain)) < tol  # two fp32 K-sum orders
    # residual epilogue in place
    r = torch.randn(M, N, device="cuda")
    r0 = r.clone()
    out = K.gemm(xt, 0, wt, 0, M, N, K_, epi=K.EPI_ADD_F32, R=r, out=r)
    assert _nerr(_np(out), _np(r0) + x @ w.T) < 1e-5 * max(1.0, (K_ / 1024) ** 0.5)


def test_split_shapes_cover_the_split(K):
    """The layouts test really runs split and unsplit shapes."""
    flags = [_splits(M, N, K_) for M, N, K_ in SHAPES]
    assert any(flags) and not all(flags)


@pytest.mark.parametrize("hd,nh,nkv,seq,B,h", [(128, 8, 2, 500, 2, 8192), (64, 8, 8, 300, 1, 8256)])
def test_split_gemm_qkv_rope(K, split, hd, nh, nkv, seq, B, h):
    rng = np.random.default_rng(hd + seq + h)
    cfg = oracle.Config(1, nh * hd, nh, nkv, 8, 8, seq, B)
    cos, sin = om.rope_tables(cfg, np.float64)
    cs = torch.tensor(np.stack([cos, sin], axis=-1).astype(np.float32)).cuda()
    T, n = B * seq, (nh + 2 * nkv) * hd
    assert _splits(T, n, h)
    a, at = _bf16(rng, (T, h))
    w, wt = _bf16(rng, (n, h), 0.05)
    got = _np(K.gemm_qkv_rope(at, wt, cs, seq, nh, nkv, hd))
    y = a @ w.T
    q = y[:, : nh * hd].reshape(B, seq, nh, hd)
    k = y[:, nh * hd:(nh + nkv) * hd].reshape(B, seq, nkv, hd)
    assert _nerr(got[:, : nh * hd], om.rope(q, cos, sin).reshape(T, -1)) < 4e-3
    assert _nerr(got[:, nh * hd:(nh + nkv) * hd], om.rope(k, cos, sin).reshape(T, -1)) < 4e-3
    assert _nerr(got[:, (nh + nkv) * hd:], y[:, (nh + nkv) * hd:]) < 4e-3


@pytest.mark.parametrize("T,h,f", [(1000, 8192, 1024), (512, 8320, 1400)])
def test_split_gemm_swiglu(K, split, T, h, f):
    rng = np.random.default_rng(T + f)
    assert _splits(T, f, h, paired=True)
    b, bt = _bf16(rng, (T, h))
    wgu, wt = _bf16(rng, (2 * f, h), 0.1)
    act, gu = K.gemm_swiglu(bt, wt, f, keep_gu=True)
    g = b @ wgu[:f].T
    u = b @ wgu[f:].T
    got_gu = _np(gu)
    assert _nerr(got_gu[:, :f], g) < 4e-3
    assert _nerr(got_gu[:, f:], u) < 4e-3
    assert _nerr(_np(act), om.swiglu(g, u)) < 8e-3


@pytest.mark.parametrize("T,h,f", [(1000, 8192, 1024), (640, 8256, 2560)])
def test_split_gemm_swiglu_bwd(K, split, T, h, f):
    rng = np.random.default_rng(3 * T + f)
    assert _splits(T, f, h)
    dy, dyt = _bf16(rng, (T, h))
    wd, wdt = _bf16(rng, (h, f), 0.05)
    gu, gut = _bf16(rng, (T, 2 * f), 2.0)
    dgu = _np(K.gemm_swiglu_bwd(dyt, wdt, gut, f))
    rdg, rdu = om.swiglu_backward(dy @ wd, gu[:, :f], gu[:, f:])
    assert _nerr(dgu[:, :f], rdg) < 4e-3
    assert _nerr(dgu[:, f:], rdu) < 4e-3


def test_split_workspace_rejects_misaligned(K):
    from host_memory_streamed_stream_gb300 import _lib

    ws = torch.zeros(64, dtype=torch.uint8, device="cuda")
    assert _lib.load().mtk_gemm_use_workspace(ws.data_ptr() + 4) == -1
    assert _lib.load().mtk_gemm_use_workspace(None) == 0
