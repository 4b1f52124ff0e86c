"""Pin the oracle's forward pieces to closed forms, special cases and brute force."""
import math

import numpy as np

import oracle
import synth
from oracle import model as om

TINY = oracle.Config(n_layers=2, hidden=256, n_heads=4, n_kv_heads=4, ffn=1024, vocab=1024, seq=128, batch=2)


def _tiny_inputs():
    W = oracle.init_params(TINY, synth, synth.WEIGHT_SEED)
    return W, synth.tokens(TINY.tokens, TINY.vocab), synth.labels(TINY.tokens, TINY.vocab)


def test_initial_loss_near_log_vocab():
    """With unit gains the normalised rows have sum(y^2) = h, so logits ~ N(0, 4e-4 h) and
    E[loss] = ln V + sigma^2 / 2 = ln V + 2e-4 h (6.983 for V = 1024, h = 256)."""
    W, tok, lab = _tiny_inputs()
    loss = oracle.loss_only(TINY, W, tok, lab)
    expect = math.log(TINY.vocab) + 2e-4 * TINY.hidden
    assert abs(loss - expect) / expect < 0.02, (loss, expect)


def test_zero_head_gives_log_vocab_exactly():
    """All-zero LM head: every logit is 0, loss = ln V, dlogits = (1/V - onehot)/T, dW_head = dz^T y."""
    W, tok, lab = _tiny_inputs()
    W[-1]["w_head"] = np.zeros_like(W[-1]["w_head"])
    loss, grads, inter = oracle.forward_backward(TINY, W, tok, lab, keep=True)
    assert abs(loss - math.log(TINY.vocab)) < 1e-12
    T, V = TINY.tokens, TINY.vocab
    dz = np.full((T, V), 1.0 / V)
    dz[np.arange(T), lab] -= 1.0
    dz /= T
    y, _ = om.rmsnorm(inter["x_final"], 1.0, TINY.rms_eps)
    np.testing.assert_allclose(grads[-1]["w_head"], dz.T @ y, rtol=0, atol=1e-12)
    # nothing flows below the head when W_head = 0
    assert np.max(np.abs(grads[0]["emb"])) == 0.0


def test_attention_single_position_returns_v():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((2, 1, 4, 16))
    k = rng.standard_normal((2, 1, 2, 16))
    v = rng.standard_normal((2, 1, 2, 16))
    o, _ = om.causal_attention(q, k, v)
    np.testing.assert_array_equal(o, np.repeat(v, 2, axis=2))


def test_attention_matches_brute_force_loops():
    """Scalar loops straight from the definition (max-free softmax in float64)."""
    rng = np.random.default_rng(1)
    B, s, nh, nkv, hd = 1, 7, 4, 2, 8
    q = rng.standard_normal((B, s, nh, hd))
    k = rng.standard_normal((B, s, nkv, hd))
    v = rng.standard_normal((B, s, nkv, hd))
    o, _ = om.causal_attention(q, k, v)
    for n in range(nh):
        kv = n // (nh // nkv)
        for i in range(s):
            w = [math.exp(sum(q[0, i, n, d] * k[0, j, kv, d] for d in range(hd)) / math.sqrt(hd))
                 for j in range(i + 1)]
            z = sum(w)
            for d in range(hd):
                ref = sum(w[j] * v[0, j, kv, d] for j in range(i + 1)) / z
                assert abs(o[0, i, n, d] - ref) < 1e-12


def test_gqa_equals_mha_with_repeated_kv():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((2, 9, 6, 8))
    k = rng.standard_normal((2, 9, 2, 8))
    v = rng.standard_normal((2, 9, 2, 8))
    o_gqa, _ = om.causal_attention(q, k, v)
    o_mha, _ = om.causal_attention(q, np.repeat(k, 3, axis=2), np.repeat(v, 3, axis=2))
    np.testing.assert_allclose(o_gqa, o_mha, rtol=0, atol=1e-14)


def test_rmsnorm_unit_mean_square():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 64)) * 3.0
    y, r = om.rmsnorm(x, np.ones(64), 0.0)
    np.testing.assert_allclose(np.mean(y * y, axis=1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(r[:, 0], 1.0 / np.sqrt(np.mean(x * x, axis=1)), rtol=1e-14)


def test_rope_properties():
    """Position 0 is the identity; each (i, i+hd/2) pair keeps its norm; the rotated
    dot product depends only on the position difference; i = 0 rotates by pos radians."""
    cfg = oracle.Config(n_layers=1, hidden=64, n_heads=4, n_kv_heads=4, ffn=8, vocab=8, seq=40, batch=1)
    cos, sin = om.rope_tables(cfg, np.float64)
    hd = cfg.head_dim
    rng = np.random.default_rng(4)
    x = rng.standard_normal((1, cfg.seq, 1, hd))
    y = om.rope(x, cos, sin)
    np.testing.assert_allclose(y[0, 0], x[0, 0], rtol=0, atol=0)
    half = hd // 2
    n_x = x[..., :half] ** 2 + x[..., half:] ** 2
    n_y = y[..., :half] ** 2 + y[..., half:] ** 2
    np.testing.assert_allclose(n_y, n_x, rtol=1e-13)
    assert abs(cos[7, 0] - math.cos(7.0)) < 1e-15 and abs(sin[7, 0] - math.sin(7.0)) < 1e-15
    assert abs(cos[5, 1] - math.cos(5.0 * 10000.0 ** (-2.0 / hd))) < 1e-15
    qv = rng.standard_normal(hd)
    kv = rng.standard_normal(hd)
    Q = om.rope(np.broadcast_to(qv, (1, cfg.seq, 1, hd)).copy(), cos, sin)[0, :, 0]
    K = om.rope(np.broadcast_to(kv, (1, cfg.seq, 1, hd)).copy(), cos, sin)[0, :, 0]
    assert abs(Q[10] @ K[4] - Q[30] @ K[24]) < 1e-12
    # backward is the transpose: <rope(x), d> == <x, rope_backward(d)>
    d = rng.standard_normal(y.shape)
    assert abs(np.sum(y * d) - np.sum(x * om.rope_backward(d, cos, sin))) < 1e-12


def test_cross_entropy_gradient_rows_sum_to_zero():
    W, tok, lab = _tiny_inputs()
    _, grads, inter = oracle.forward_backward(TINY, W, tok, lab, keep=True)
    # dW_head^T = y^T dz: the columns of dW_head sum, over vocab, to y^T (sum_v dz) = 0
    np.testing.assert_allclose(grads[-1]["w_head"].sum(axis=0), 0.0, atol=1e-15)


def test_silu_values():
    assert om.silu(np.array(0.0)) == 0.0
    assert abs(om.silu(np.array(1.0)) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    assert abs(om.silu(np.array(-30.0))) < 1e-11


def test_embedding_gradient_is_ordered_scatter():
    """Every row of dE equals the sum of dx0 over the positions holding that token."""
    W, tok, lab = _tiny_inputs()
    _, grads, inter = oracle.forward_backward(TINY, W, tok, lab, keep=True)
    dx0 = inter["dx0"]
    for v in [int(tok[0]), int(tok[17]), 5]:
        idx = np.nonzero(tok == v)[0]
        ref = dx0[idx].sum(axis=0) if idx.size else np.zeros(TINY.hidden)
        np.testing.assert_allclose(grads[0]["emb"][v], ref, rtol=1e-13, atol=1e-18)
    unused = np.setdiff1d(np.arange(TINY.vocab), tok)
    assert np.all(grads[0]["emb"][unused] == 0)


def test_row_wise_attention_equals_the_full_matrix():
    """The row-wise forms (used where an s x s matrix cannot be held) give what the full-matrix
    attention and its backward give, head by head, in float64; GQA heads share k and v."""
    rng = np.random.default_rng(5)
    B, s, nh, nkv, hd = 1, 300, 4, 2, 32
    q = rng.standard_normal((B, s, nh, hd)) * 2.0
    k = rng.standard_normal((B, s, nkv, hd))
    v = rng.standard_normal((B, s, nkv, hd))
    do = rng.standard_normal((B, s, nh, hd))
    o, P = om.causal_attention(q, k, v)
    dq, dk, dv = om.causal_attention_backward(do, q, k, v, P)
    dk_rows, dv_rows = np.zeros_like(dk), np.zeros_like(dv)
    for n in range(nh):
        kv = n // (nh // nkv)
        o_n, lse_n = om.causal_attention_all_rows(q[0, :, n], k[0, :, kv], v[0, :, kv], chunk=64)
        np.testing.assert_allclose(o_n, o[0, :, n], rtol=0, atol=1e-12)
        # lse against its definition on a few rows
        for i in (0, 1, 77, s - 1):
            sc = q[0, i, n] @ k[0, : i + 1, kv].T / math.sqrt(hd)
            assert abs(lse_n[i] - math.log(np.sum(np.exp(sc)))) < 1e-12
        sel = np.array([0, 5, 64, 299])
        o_sel, _ = om.causal_attention_rows(q[0, :, n], k[0, :, kv], v[0, :, kv], sel)
        np.testing.assert_allclose(o_sel, o[0, sel, n], rtol=0, atol=1e-12)
        dq_n, dk_n, dv_n = om.causal_attention_backward_rows(do[0, :, n], q[0, :, n], k[0, :, kv], v[0, :, kv],
                                                             o_n, lse_n, chunk=64)
        np.testing.assert_allclose(dq_n, dq[0, :, n], rtol=0, atol=1e-11)
        dk_rows[0, :, kv] += dk_n
        dv_rows[0, :, kv] += dv_n
        # the sampled forms: dq of listed query rows, dk/dv of listed key positions
        D = np.sum(do[0, :, n] * o_n, axis=1)
        dq_sel = om.causal_attention_dq_rows(do[0, :, n], q[0, :, n], k[0, :, kv], v[0, :, kv], lse_n, D, sel)
        np.testing.assert_allclose(dq_sel, dq_n[sel], rtol=0, atol=1e-11)
        dk_sel, dv_sel = om.causal_attention_dkv_cols(do[0, :, n], q[0, :, n], k[0, :, kv], v[0, :, kv], lse_n, D,
                                                      sel)
        np.testing.assert_allclose(dk_sel, dk_n[sel], rtol=0, atol=1e-11)
        np.testing.assert_allclose(dv_sel, dv_n[sel], rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk_rows, dk, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv_rows, dv, rtol=0, atol=1e-11)
