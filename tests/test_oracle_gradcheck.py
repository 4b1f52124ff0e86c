"""Pin the oracle's backward pass to its forward pass with float64 central differences.

The analytic gradient of every parameter kind (every gain in full, sampled
coordinates of every matrix and of the embedding) must match
(L(p + e) - L(p - e)) / 2e. A dropped term, a wrong sign or a transposed
operand anywhere in the backward pass shows up as an O(1) relative error.
The mutation tests at the end plant such mistakes in the oracle (on the CPU,
by monkeypatching) and check that this comparison catches them.
"""
import numpy as np
import pytest

import oracle
from oracle import model as om

MICRO = oracle.Config(n_layers=2, hidden=32, n_heads=4, n_kv_heads=2, ffn=48, vocab=40, seq=8, batch=2)
TINY = oracle.Config(n_layers=2, hidden=256, n_heads=4, n_kv_heads=4, ffn=1024, vocab=1024, seq=128, batch=2)


def _random_float_params(cfg, seed, std=0.3):
    """float64 weights with O(1) activations, so every nonlinearity is exercised."""
    rng = np.random.default_rng(seed)
    out = []
    for b in range(cfg.n_layers + 2):
        d = {}
        for name, shape in om.block_tensors(cfg, b):
            if len(shape) == 1:
                d[name] = 1.0 + 0.3 * rng.standard_normal(shape)
            else:
                d[name] = std * rng.standard_normal(shape)
        out.append(d)
    return out


def _coords(shape, rng, n_matrix, n_gain=None):
    if len(shape) == 1 and (n_gain is None or n_gain >= shape[0]):
        return [(i,) for i in range(shape[0])]
    if len(shape) == 1:
        return [(int(i),) for i in rng.choice(shape[0], size=n_gain, replace=False)]
    flat = rng.choice(int(np.prod(shape)), size=min(n_matrix, int(np.prod(shape))), replace=False)
    return [tuple(int(c) for c in np.unravel_index(f, shape)) for f in flat]


def _fd_errors(cfg, W, tok, lab, n_matrix, seed=0, eps_rel=1e-5, only=None, n_gain=None):
    """max |fd - analytic| / max|analytic| per tensor kind."""
    _, grads = oracle.forward_backward(cfg, W, tok, lab, np.float64)
    rng = np.random.default_rng(seed)
    errs = {}
    for b in range(cfg.n_layers + 2):
        for name, shape in om.block_tensors(cfg, b):
            if only is not None and name not in only:
                continue
            g = grads[b][name]
            scale = np.max(np.abs(g))
            worst = 0.0
            for c in _coords(shape, rng, n_matrix, n_gain):
                p0 = W[b][name][c]
                eps = eps_rel * max(1.0, abs(p0))
                W[b][name][c] = p0 + eps
                lp = oracle.loss_only(cfg, W, tok, lab)
                W[b][name][c] = p0 - eps
                lm = oracle.loss_only(cfg, W, tok, lab)
                W[b][name][c] = p0
                fd = (lp - lm) / (2 * eps)
                worst = max(worst, abs(fd - g[c]) / scale)
            errs[(b, name)] = worst
    return errs


def _micro_inputs(seed=3):
    rng = np.random.default_rng(seed)
    tok = rng.integers(0, MICRO.vocab, MICRO.tokens)
    lab = rng.integers(0, MICRO.vocab, MICRO.tokens)
    return tok, lab


def test_fd_micro_all_kinds():
    """GQA micro model: every gain coordinate and 48 coordinates of every matrix."""
    W = _random_float_params(MICRO, 11)
    tok, lab = _micro_inputs()
    errs = _fd_errors(MICRO, W, tok, lab, n_matrix=48)
    bad = {k: v for k, v in errs.items() if v > 1e-6}
    assert not bad, bad


def test_fd_tiny_config_sampled():
    """The tiny benchmark shape (head_dim 64, seq 128) at its real init scale: sampled coordinates."""
    import synth

    Wb = oracle.init_params(TINY, synth, synth.WEIGHT_SEED)
    W = [{k: om.bf16_bits_to_float(v) for k, v in blk.items()} for blk in Wb]
    tok = synth.tokens(TINY.tokens, TINY.vocab)
    lab = synth.labels(TINY.tokens, TINY.vocab)
    errs = _fd_errors(TINY, W, tok, lab, n_matrix=6, seed=1, eps_rel=1e-4,
                      n_gain=6)
    bad = {k: v for k, v in errs.items() if v > 1e-6}
    assert not bad, bad


def test_float32_oracle_close_to_float64():
    """The float32 instantiation agrees with float64 to float32 accuracy."""
    import synth

    Wb = oracle.init_params(TINY, synth, synth.WEIGHT_SEED)
    tok = synth.tokens(TINY.tokens, TINY.vocab)
    lab = synth.labels(TINY.tokens, TINY.vocab)
    l64, g64 = oracle.forward_backward(TINY, Wb, tok, lab, np.float64)
    l32, g32 = oracle.forward_backward(TINY, Wb, tok, lab, np.float32)
    assert abs(l32 - l64) / l64 < 1e-5
    for b in range(TINY.n_layers + 2):
        for k in g64[b]:
            err = np.max(np.abs(g32[b][k] - g64[b][k])) / np.max(np.abs(g64[b][k]))
            assert err < 1e-4, (b, k, err)


# ---------------------------------------------------------------------------
# planted mistakes: each must be caught by the comparison above
# ---------------------------------------------------------------------------
def _planted(monkeypatch, attr, fn):
    monkeypatch.setattr(om, attr, fn)
    W = _random_float_params(MICRO, 11)
    tok, lab = _micro_inputs()
    errs = _fd_errors(MICRO, W, tok, lab, n_matrix=16)
    return max(errs.values())


def test_planted_rmsnorm_term_dropped(monkeypatch):
    def bad(dy, x, gamma, r):
        xhat = x * r
        return r * dy * gamma, np.sum(dy * xhat, axis=0)  # drops the projection term
    assert _planted(monkeypatch, "rmsnorm_backward", bad) > 1e-2


def test_planted_rope_sign(monkeypatch):
    def bad(dy, cos, sin):
        half = dy.shape[-1] // 2
        d1, d2 = dy[..., :half], dy[..., half:]
        c, s = cos[None, :, None, :], sin[None, :, None, :]
        return np.concatenate([d1 * c - d2 * s, d2 * c + d1 * s], axis=-1)  # forward rotation
    assert _planted(monkeypatch, "rope_backward", bad) > 1e-2


def test_planted_attention_transpose(monkeypatch):
    orig = om.causal_attention_backward

    def bad(do, q, k, v, P):
        dq, dk, dv = orig(do, q, k, v, P)
        return dq, dk, np.swapaxes(dv, 1, 1)[:, ::-1]  # positions reversed
    assert _planted(monkeypatch, "causal_attention_backward", bad) > 1e-2
