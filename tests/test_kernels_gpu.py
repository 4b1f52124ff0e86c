"""Each layer-template kernel, through the C ABI, against the oracle's op on the same inputs.

Shapes span several tiles and ragged tails. Tolerances: fp32 results within
fp32-accumulation error of the float64 oracle; bf16 results within 2e-2 of the
tensor's max magnitude (the stated gradient bar), most far tighter.
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


def _bf16(rng, shape, scale=1.0):
    """bf16 values (as a float64 numpy array) and the matching torch tensor on the GPU."""
    x = oracle.bf16_bits_to_float(oracle.float_to_bf16_bits(rng.standard_normal(shape) * scale))
    return x, torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).cuda()


def _f32(rng, shape, scale=1.0):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    return x.astype(np.float64), torch.tensor(x).cuda()


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


def _nerr(got, ref):
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))


@pytest.mark.parametrize("M,N,K_", [(1000, 776, 328), (128, 256, 64), (4096, 2048, 1024), (8, 8, 8)])
def test_gemm_three_layouts(K, M, N, K_):
    rng = np.random.default_rng(M + N + K_)
    x, xt = _bf16(rng, (M, K_))
    w, wt = _bf16(rng, (N, K_))
    ref = x @ w.T
    # forward: A [M][K], B [N][K]
    y = K.gemm(xt, 0, wt, 0, M, N, K_, epi=K.EPI_STORE_F32)
    assert _nerr(_np(y), ref) < 1e-5
    yb = K.gemm(xt, 0, wt, 0, M, N, K_, epi=K.EPI_STORE_BF16)
    assert _nerr(_np(yb), ref) < 4e-3
    # dgrad: dX[M][K] = dY[M][N] W[N][K]  (B stored [K=N][N=K], MN-major)
    dy, dyt = _bf16(rng, (M, N))
    dx = K.gemm(dyt, 0, wt, 1, M, K_, N, epi=K.EPI_STORE_F32)
    assert _nerr(_np(dx), dy @ w) < 1e-5
    # wgrad: dW[N][K] = dY^T X  (A stored [T=M][N], B stored [T=M][K], both MN-major)
    dw = K.gemm(dyt, 1, xt, 1, N, K_, M, epi=K.EPI_STORE_F32)
    assert _nerr(_np(dw), dy.T @ x) < 1e-5
    # residual epilogue, in place
    r, rt = _f32(rng, (M, N))
    out = K.gemm(xt, 0, wt, 0, M, N, K_, epi=K.EPI_ADD_F32, R=rt, out=rt)
    assert out.data_ptr() == rt.data_ptr()
    assert _nerr(_np(out), r + ref) < 1e-5


def test_gemm_deterministic(K):
    rng = np.random.default_rng(5)
    _, at = _bf16(rng, (2048, 1536))
    _, bt = _bf16(rng, (2048, 1024))
    c1 = K.gemm(at, 1, bt, 1, 1536, 1024, 2048, epi=K.EPI_STORE_F32)
    c2 = K.gemm(at, 1, bt, 1, 1536, 1024, 2048, epi=K.EPI_STORE_F32)
    assert torch.equal(c1, c2)


# (more rows than the backward's 304 parts: each CTA streams several rows through its ring)
@pytest.mark.parametrize("T,h", [(300, 256), (64, 4096), (33, 5120), (3000, 4096), (2000, 5120), (5000, 2048)])
def test_rmsnorm_forward_backward(K, T, h):
    rng = np.random.default_rng(T + h)
    x, xt = _f32(rng, (T, h), 2.0)
    g, gt = _bf16(rng, (h,), 0.5)
    g = g + 1.0
    gt = gt.float().add(1.0).to(torch.bfloat16)
    g = _np(gt)
    y, rstd = K.rmsnorm_fwd(xt, gt, 1e-5)
    ref, r = om.rmsnorm(x, g, 1e-5)
    assert _nerr(_np(rstd), r[:, 0]) < 1e-6
    assert _nerr(_np(y), ref) < 4e-3
    dy, dyt = _f32(rng, (T, h))
    dres, drt = _f32(rng, (T, h))
    dx, dxb, dg = K.rmsnorm_bwd(dyt, xt, gt, rstd, drt)
    rdx, rdg = om.rmsnorm_backward(dy, x, g, r)
    assert _nerr(_np(dx), rdx + dres) < 1e-5
    assert _nerr(_np(dxb), rdx + dres) < 4e-3
    assert _nerr(_np(dg), rdg) < 4e-3


@pytest.mark.parametrize("limit_ms", [1, 20])
def test_bounded_wait_gives_up_and_the_context_stays_usable(K, limit_ms):
    """A wait that can never be satisfied (an mbarrier nobody arrives on) gives up after its
    limit through the same routine the GEMM and attention pipelines use: it records code 6 in
    the error flag and returns. The next kernels then run normally."""
    import time

    from host_memory_streamed_stream_gb300 import _lib

    lib = _lib.load()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gave_up = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert lib.mtk_bounded_wait_check(err.data_ptr(), gave_up.data_ptr(), limit_ms * 1_000_000, None) == 0
    torch.cuda.synchronize()
    el = time.perf_counter() - t0
    assert int(err.item()) == 6 and int(gave_up.item()) == 1
    assert limit_ms * 1e-3 <= el < 5.0
    # a flag already set makes the wait give up at once, leaving the first code in place
    gave_up.zero_()
    assert lib.mtk_bounded_wait_check(err.data_ptr(), gave_up.data_ptr(), 4_000_000_000, None) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 6 and int(gave_up.item()) == 1
    assert lib.mtk_bounded_wait_check(err.data_ptr(), gave_up.data_ptr(), -1, None) == -1
    # the context is fine: a GEMM afterwards is exact against the oracle's product
    rng = np.random.default_rng(7)
    x, xt = _bf16(rng, (256, 128))
    w, wt = _bf16(rng, (192, 128))
    y = K.gemm(xt, 0, wt, 0, 256, 192, 128, epi=K.EPI_STORE_F32)
    assert _nerr(_np(y), x @ w.T) < 1e-5


def test_rmsnorm_rejects_misaligned_pointers(K):
    """An fp32 row slice at an odd offset (or an 8-byte-misaligned bf16 gain) is rejected with
    MT_EINVAL before any launch, so the vector accesses never see it."""
    from host_memory_streamed_stream_gb300 import _lib

    lib = _lib.load()
    T, h = 16, 512
    buf = torch.zeros(T + 1, h, device="cuda")
    g = torch.ones(h + 8, dtype=torch.bfloat16, device="cuda")
    rstd = torch.ones(T, device="cuda")
    part = torch.zeros(lib.mtk_rmsnorm_bwd_parts(T) + 1, h, device="cuda")
    dg = torch.empty(h, dtype=torch.bfloat16, device="cuda")
    p, gp = buf.data_ptr(), g.data_ptr()
    for dy, x, gam, dx, pt in ((p + 4, p, gp, p, part.data_ptr()), (p, p + 8, gp, p, part.data_ptr()),
                               (p, p, gp + 2, p, part.data_ptr()), (p, p, gp, p + 12, part.data_ptr()),
                               (p, p, gp, p, part.data_ptr() + 4)):
        rc = lib.mtk_rmsnorm_bwd(dy, x, gam, rstd.data_ptr(), None, dx, None, pt, dg.data_ptr(), T, h, None)
        assert rc == -1
        assert b"aligned" in lib.mt_last_error(None)
    y = torch.empty(T, h, dtype=torch.bfloat16, device="cuda")
    assert lib.mtk_rmsnorm_fwd(p + 4, gp, y.data_ptr(), rstd.data_ptr(), T, h, 1e-5, None) == -1
    assert lib.mtk_rmsnorm_fwd(p, gp + 2, y.data_ptr(), rstd.data_ptr(), T, h, 1e-5, None) == -1
    torch.cuda.synchronize()


@pytest.mark.parametrize("hd,nh,nkv,seq,B", [(64, 4, 4, 128, 2), (128, 8, 2, 200, 2)])
def test_rope_forward_inverse(K, hd, nh, nkv, seq, B):
    rng = np.random.default_rng(hd + seq)
    cfg = oracle.Config(1, nh * hd, nh, nkv, 8, 8, seq, B)
    cos, sin = om.rope_tables(cfg, np.float64)
    cs = torch.tensor(np.stack([cos, sin], axis=-1).astype(np.float32)).cuda()
    ld = (nh + 2 * nkv) * hd
    qkv, qt = _bf16(rng, (B * seq, ld))
    K.rope_(qt, seq, nh, nkv, hd, cs)
    got = _np(qt)
    q = qkv[:, : nh * hd].reshape(B, seq, nh, hd)
    k = qkv[:, nh * hd:(nh + nkv) * hd].reshape(B, seq, nkv, hd)
    assert _nerr(got[:, : nh * hd], om.rope(q, cos, sin).reshape(B * seq, -1)) < 4e-3
    assert _nerr(got[:, nh * hd:(nh + nkv) * hd], om.rope(k, cos, sin).reshape(B * seq, -1)) < 4e-3
    np.testing.assert_array_equal(got[:, (nh + nkv) * hd:], qkv[:, (nh + nkv) * hd:])  # v untouched
    d, dt = _bf16(rng, (B * seq, ld))
    K.rope_(dt, seq, nh, nkv, hd, cs, inverse=True)
    dq = d[:, : nh * hd].reshape(B, seq, nh, hd)
    assert _nerr(_np(dt)[:, : nh * hd], om.rope_backward(dq, cos, sin).reshape(B * seq, -1)) < 4e-3


@pytest.mark.parametrize("T,f", [(300, 1368), (64, 11008)])
def test_swiglu(K, T, f):
    rng = np.random.default_rng(f)
    gu, gut = _bf16(rng, (T, 2 * f), 2.0)
    act = K.swiglu_fwd(gut, f)
    g, u = gu[:, :f], gu[:, f:]
    assert _nerr(_np(act), om.swiglu(g, u)) < 4e-3
    da, dat = _bf16(rng, (T, f))
    dgu = _np(K.swiglu_bwd(gut, dat, f))
    rdg, rdu = om.swiglu_backward(da, g, u)
    assert _nerr(dgu[:, :f], rdg) < 4e-3
    assert _nerr(dgu[:, f:], rdu) < 4e-3



@pytest.mark.parametrize("hd,nh,nkv,seq,B,h", [(64, 4, 4, 128, 2, 256), (128, 8, 2, 200, 2, 512), (128, 2, 1, 70, 1, 64)])
def test_gemm_qkv_rope_fused(K, hd, nh, nkv, seq, B, h):
    """QKV projection with RoPE in the epilogue vs the oracle's projection then rotation."""
    rng = np.random.default_rng(hd + seq + h)
    cfg = oracle.Config(1, nh * hd, nh, nkv, 8, 8, seq, B)
    cos, sin = om.rope_tables(cfg, np.float64)
    cs = torch.tensor(np.stack([cos, sin], axis=-1).astype(np.float32)).cuda()
    T, n = B * seq, (nh + 2 * nkv) * hd
    a, at = _bf16(rng, (T, h))
    w, wt = _bf16(rng, (n, h), 0.05)
    got = _np(K.gemm_qkv_rope(at, wt, cs, seq, nh, nkv, hd))
    y = a @ w.T
    q = y[:, : nh * hd].reshape(B, seq, nh, hd)
    k = y[:, nh * hd:(nh + nkv) * hd].reshape(B, seq, nkv, hd)
    assert _nerr(got[:, : nh * hd], om.rope(q, cos, sin).reshape(T, -1)) < 4e-3
    assert _nerr(got[:, nh * hd:(nh + nkv) * hd], om.rope(k, cos, sin).reshape(T, -1)) < 4e-3
    assert _nerr(got[:, (nh + nkv) * hd:], y[:, (nh + nkv) * hd:]) < 4e-3


@pytest.mark.parametrize("T,h,f", [(300, 256, 1368), (256, 512, 11008), (130, 64, 72)])
def test_gemm_swiglu_fused(K, T, h, f):
    """Gate-up projection with SwiGLU in the epilogue: act, and [g | u] when kept."""
    rng = np.random.default_rng(T + f)
    b, bt = _bf16(rng, (T, h))
    wgu, wt = _bf16(rng, (2 * f, h), 0.1)
    act, gu = K.gemm_swiglu(bt, wt, f, keep_gu=True)
    act_only, none = K.gemm_swiglu(bt, wt, f)
    assert none is None and torch.equal(act, act_only)
    g = b @ wgu[:f].T
    u = b @ wgu[f:].T
    got_gu = _np(gu)
    assert _nerr(got_gu[:, :f], g) < 4e-3
    assert _nerr(got_gu[:, f:], u) < 4e-3
    assert _nerr(_np(act), om.swiglu(g, u)) < 8e-3


@pytest.mark.parametrize("T,h,f", [(300, 256, 1368), (200, 4096, 512), (130, 64, 72)])
def test_gemm_swiglu_bwd_fused(K, T, h, f):
    """Down-projection data gradient with the SwiGLU backward in the epilogue."""
    rng = np.random.default_rng(3 * T + f)
    dy, dyt = _bf16(rng, (T, h))
    wd, wdt = _bf16(rng, (h, f), 0.05)
    gu, gut = _bf16(rng, (T, 2 * f), 2.0)
    dgu = _np(K.gemm_swiglu_bwd(dyt, wdt, gut, f))
    rdg, rdu = om.swiglu_backward(dy @ wd, gu[:, :f], gu[:, f:])
    assert _nerr(dgu[:, :f], rdg) < 4e-3
    assert _nerr(dgu[:, f:], rdu) < 4e-3

def test_embedding_gather_and_ordered_scatter(K):
    rng = np.random.default_rng(7)
    V, h, T = 1000, 512, 777
    E, Et = _bf16(rng, (V, h))
    tok = rng.integers(0, 60, T).astype(np.int32)  # many repeats
    x = K.embed_fwd(torch.tensor(tok).cuda(), Et)
    np.testing.assert_array_equal(_np(x), E[tok])
    dx, dxt = _f32(rng, (T, h))
    order = np.argsort(tok, kind="stable").astype(np.int32)
    offsets = np.concatenate([[0], np.cumsum(np.bincount(tok, minlength=V))]).astype(np.int32)
    dE = K.embed_bwd(torch.tensor(order).cuda(), torch.tensor(offsets).cuda(), dxt, V)
    ref = om.embedding_backward(dx, tok, V)
    assert _nerr(_np(dE), ref) < 4e-3
    assert np.all(_np(dE)[60:] == 0)


@pytest.mark.parametrize("T,V", [(300, 1000), (64, 152064)])
def test_cross_entropy(K, T, V):
    rng = np.random.default_rng(V)
    z, zt = _f32(rng, (T, V), 3.0)
    lab = rng.integers(0, V, T).astype(np.int32)
    loss, rows, dl = K.cross_entropy(zt, torch.tensor(lab).cuda())
    rrows, rdz = om.cross_entropy(z, lab)
    assert _nerr(_np(rows), rrows) < 1e-5
    assert abs(loss.item() - rrows.mean()) < 1e-5 * abs(rrows.mean())
    assert _nerr(_np(dl), rdz) < 4e-3


def test_cross_entropy_zero_logits_exact(K):
    T, V = 40, 1024
    z = torch.zeros(T, V, device="cuda")
    lab = torch.arange(T, dtype=torch.int32, device="cuda")
    loss, rows, dl = K.cross_entropy(z, lab)
    assert abs(loss.item() - np.log(V)) < 1e-6


@pytest.mark.parametrize("B,s,nh,nkv,hd", [(2, 128, 4, 4, 64), (2, 200, 4, 2, 128), (1, 1, 2, 1, 64),
                                           (1, 130, 8, 8, 128), (1, 600, 8, 2, 128), (2, 333, 4, 1, 64)])
def test_attention_forward_backward(K, B, s, nh, nkv, hd):
    rng = np.random.default_rng(s + nh)
    ld = (nh + 2 * nkv) * hd
    qkv, qkvt = _bf16(rng, (B * s, ld))
    o, lse = K.attn_fwd(qkvt, B, s, nh, nkv, hd)
    q = qkv[:, : nh * hd].reshape(B, s, nh, hd)
    k = qkv[:, nh * hd:(nh + nkv) * hd].reshape(B, s, nkv, hd)
    v = qkv[:, (nh + nkv) * hd:].reshape(B, s, nkv, hd)
    ro, P = om.causal_attention(q, k, v)
    assert _nerr(_np(o), ro.reshape(B * s, -1)) < 1e-2
    if s == 1:  # one position: the output is v (per query head's kv head)
        np.testing.assert_allclose(_np(o).reshape(B, 1, nh, hd), np.repeat(v, nh // nkv, axis=2), atol=1e-2)
    do, dot = _bf16(rng, (B * s, nh * hd))
    dqkv = _np(K.attn_bwd(qkvt, o, lse, dot, B, s, nh, nkv, hd))
    rdq, rdk, rdv = om.causal_attention_backward(do.reshape(B, s, nh, hd), q, k, v, P)
    assert _nerr(dqkv[:, : nh * hd], rdq.reshape(B * s, -1)) < 2e-2
    assert _nerr(dqkv[:, nh * hd:(nh + nkv) * hd], rdk.reshape(B * s, -1)) < 2e-2
    assert _nerr(dqkv[:, (nh + nkv) * hd:], rdv.reshape(B * s, -1)) < 2e-2



@pytest.mark.parametrize("B,s,nh,nkv,hd", [(2, 200, 4, 2, 128), (1, 333, 4, 4, 64)])
def test_attention_backward_with_rope(K, B, s, nh, nkv, hd):
    """dq/dk from the fused backward equal the oracle's attention backward followed by its
    RoPE backward; dv is untouched by the rotation."""
    rng = np.random.default_rng(7 * s + hd)
    cfg = oracle.Config(1, nh * hd, nh, nkv, 8, 8, s, B)
    cos, sin = om.rope_tables(cfg, np.float64)
    cs = torch.tensor(np.stack([cos, sin], axis=-1).astype(np.float32)).cuda()
    ld = (nh + 2 * nkv) * hd
    qkv, qkvt = _bf16(rng, (B * s, ld))
    o, lse = K.attn_fwd(qkvt, B, s, nh, nkv, hd)
    do, dot = _bf16(rng, (B * s, nh * hd))
    dqkv = _np(K.attn_bwd(qkvt, o, lse, dot, B, s, nh, nkv, hd, cos_sin=cs))
    q = qkv[:, : nh * hd].reshape(B, s, nh, hd)
    k = qkv[:, nh * hd:(nh + nkv) * hd].reshape(B, s, nkv, hd)
    v = qkv[:, (nh + nkv) * hd:].reshape(B, s, nkv, hd)
    _, P = om.causal_attention(q, k, v)
    rdq, rdk, rdv = om.causal_attention_backward(do.reshape(B, s, nh, hd), q, k, v, P)
    assert _nerr(dqkv[:, : nh * hd], om.rope_backward(rdq, cos, sin).reshape(B * s, -1)) < 2e-2
    assert _nerr(dqkv[:, nh * hd:(nh + nkv) * hd], om.rope_backward(rdk, cos, sin).reshape(B * s, -1)) < 2e-2
    assert _nerr(dqkv[:, (nh + nkv) * hd:], rdv.reshape(B * s, -1)) < 2e-2

def test_attention_deterministic(K):
    rng = np.random.default_rng(11)
    B, s, nh, nkv, hd = 1, 300, 8, 2, 128
    _, qkvt = _bf16(rng, (B * s, (nh + 2 * nkv) * hd))
    o, lse = K.attn_fwd(qkvt, B, s, nh, nkv, hd)
    _, dot = _bf16(rng, (B * s, nh * hd))
    a = K.attn_bwd(qkvt, o, lse, dot, B, s, nh, nkv, hd)
    b = K.attn_bwd(qkvt, o, lse, dot, B, s, nh, nkv, hd)
    assert torch.equal(a, b)


def test_attention_forward_output_waits_for_every_product(K):
    """With two 64-key tiles per 128-query tile (seq 128) the softmax warps finish their last
    tile while the products O += P V of the tile may still be running; the output must wait for
    all of them. Many CTAs, repeated: every run bit-identical, and equal to the oracle."""
    rng = np.random.default_rng(21)
    B, s, nh, nkv, hd = 64, 128, 16, 16, 128
    qkv, qkvt = _bf16(rng, (B * s, (nh + 2 * nkv) * hd))
    o0, lse0 = K.attn_fwd(qkvt, B, s, nh, nkv, hd)
    for _ in range(30):
        o, lse = K.attn_fwd(qkvt, B, s, nh, nkv, hd)
        assert torch.equal(o, o0) and torch.equal(lse, lse0)
    q = qkv[:, : nh * hd].reshape(B, s, nh, hd)[:4]
    k = qkv[:, nh * hd:(nh + nkv) * hd].reshape(B, s, nkv, hd)[:4]
    v = qkv[:, (nh + nkv) * hd:].reshape(B, s, nkv, hd)[:4]
    ro, _ = om.causal_attention(q, k, v)
    assert _nerr(_np(o0)[: 4 * s], ro.reshape(4 * s, -1)) < 1e-2
