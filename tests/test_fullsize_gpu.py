"""Parity at the benchmark configurations' full sizes, in the launch configuration bench.py times.

A whole-model oracle step at these sizes would take the CPU hours, so the oracle is
teacher-forced from the GPU step's own layer-boundary checkpoints (mt_read_checkpoint):

* x_0 equals the embedding rows of the tokens exactly;
* the loss, and the head's gradients (final norm, LM head), recomputed by the oracle from
  the GPU's final hidden state x_L;
* the last decoder layer's forward (x_{L-1} -> x_L) and all nine of its weight gradients,
  with the upstream gradient from the oracle's own head backward;
* the initial loss against its closed form ln V + 2e-4 h.

Bars as everywhere: loss 1e-3 relative, tensors 2e-2 of their max magnitude. The oracle runs
in float32 here (its float32 instantiation is pinned to float64 on the CPU). Host memory is
checked before each configuration; one that does not fit is skipped with the reason.
"""
import math
import os

import numpy as np
import pytest

import oracle
import synth
from oracle import model as om

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

CFGS = {
    "1.3b": dict(n_layers=24, hidden=2048, n_heads=16, n_kv_heads=16, ffn=5504, vocab=32000, seq=2048, batch=4),
    "7b": dict(n_layers=32, hidden=4096, n_heads=32, n_kv_heads=32, ffn=11008, vocab=32000, seq=4096, batch=2),
    "14b": dict(n_layers=48, hidden=5120, n_heads=40, n_kv_heads=8, ffn=13824, vocab=152064, seq=4096, batch=1),
}
LAYER_NAMES = ["attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "wg", "wu", "wd"]


@pytest.fixture(scope="module")
def mt():
    from host_memory_streamed_stream_gb300 import _build

    _build.build()
    import host_memory_streamed_stream_gb300 as m

    return m


def _mem_available():
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def _nerr(got, ref):
    return float(np.max(np.abs(got - ref)) / np.max(np.abs(ref)))


def _bits(mt, cfg, arena, block, section):
    """Copies of one block's tensors of a bf16 section (bit patterns), shaped."""
    out = {}
    for t in range(mt.num_tensors(cfg, block)):
        off, rows, cols, _ = mt.tensor_offset(cfg, block, section, t)
        v = arena.array[off:off + rows * cols * 2].view(np.uint16).copy()
        out[t] = v.reshape(rows) if cols == 1 else v.reshape(rows, cols)
    return out


def _f(bits, dtype=np.float32):
    return {k: oracle.bf16_bits_to_float(v, dtype) for k, v in bits.items()}


@pytest.mark.parametrize("name", list(CFGS))
def test_fullsize_teacher_forced(mt, name):
    kw = CFGS[name]
    cfg = mt.ModelConfig(**kw)
    need = mt.arena_bytes(cfg) + 12 * 2**30
    if _mem_available() < need:
        pytest.skip(f"host memory: {_mem_available() / 2**30:.0f} GiB available, {need / 2**30:.0f} GiB needed")
    ocfg = oracle.Config(**kw)
    L, T, V, h = cfg.n_layers, cfg.tokens, cfg.vocab, cfg.hidden
    tok = synth.tokens(T, V)
    lab = synth.labels(T, V)
    dt = np.float32
    # run the step, copy what the oracle needs (bf16 bit patterns, checkpoints), then free the
    # pinned arena before the oracle allocates its own arrays
    with mt.Trainer(cfg) as tr:
        mt.fill_synthetic(cfg, tr.arena, synth, synth.WEIGHT_SEED)
        loss = tr.step(tok, lab)
        x0 = tr.read_checkpoint(0)
        xl1 = tr.read_checkpoint(L - 1)
        xL = tr.read_checkpoint(L)
        off, _, _, _ = mt.tensor_offset(cfg, 0, mt.SEC_W, 0)
        E_rows = tr.arena.array[off:off + V * h * 2].view(np.uint16).reshape(V, h)[tok].copy()
        Wlast, Whead = _bits(mt, cfg, tr.arena, L, mt.SEC_W), _bits(mt, cfg, tr.arena, L + 1, mt.SEC_W)
        Glast, Ghead = _bits(mt, cfg, tr.arena, L, mt.SEC_G), _bits(mt, cfg, tr.arena, L + 1, mt.SEC_G)
    Wlast, Whead, Glast, Ghead = _f(Wlast), _f(Whead), _f(Glast), _f(Ghead)

    # the initial loss against its closed form (unit gains, N(0, 0.02^2) head)
    expect = math.log(V) + 2e-4 * h
    assert abs(loss - expect) / expect < 0.02, (loss, expect)
    # embedding gather: exact
    np.testing.assert_array_equal(x0, oracle.bf16_bits_to_float(E_rows, np.float32))

    # head, teacher-forced from the GPU's x_L
    ph = {"final_norm": Whead[0], "w_head": Whead[1]}
    ref_loss, dxL, gh, _ = om.head_forward_backward(xL.astype(dt), ph, lab, ocfg)
    assert abs(loss - ref_loss) <= 1e-3 * abs(ref_loss), (loss, ref_loss)
    assert _nerr(Ghead[0], gh["final_norm"]) <= 2e-2
    assert _nerr(Ghead[1], gh["w_head"]) <= 2e-2

    # last decoder layer: forward from the GPU's x_{L-1}, backward from the oracle's dL/dx_L
    p = {n: Wlast[i] for i, n in enumerate(LAYER_NAMES)}
    cos, sin = om.rope_tables(ocfg, dt)
    x_out, cache = om.layer_forward(xl1.astype(dt), p, ocfg, cos, sin)
    d_ref = x_out - xl1
    assert _nerr(xL - xl1, d_ref) <= 2e-2
    _, g = om.layer_backward(dxL, cache, p, ocfg, cos, sin)
    for i, n in enumerate(LAYER_NAMES):
        assert _nerr(Glast[i], g[n]) <= 2e-2, (n, _nerr(Glast[i], g[n]))


def test_fullsize_long_context_sampled_rows(mt):
    """7B shape at seq 131072 with checkpoints offloaded to pinned host memory.

    The oracle cannot hold 131072 x 131072 attention matrices, so layer 0 is recomputed on
    sampled query positions only: RMSNorm, q/k/v, RoPE and causal attention over every earlier
    key of those rows, the output projection, the FFN. Its x_1 rows are compared with the
    GPU's checkpoint x_1 (read back from the host copy), plus the exact embedding gather and
    the closed-form initial loss.
    """
    kw = dict(n_layers=32, hidden=4096, n_heads=32, n_kv_heads=32, ffn=11008, vocab=32000, seq=131072, batch=1)
    cfg = mt.ModelConfig(**kw, flags=mt.FLAG_OFFLOAD_CKPT)
    pinned = mt.arena_bytes(cfg) + cfg.n_layers * cfg.tokens * cfg.hidden * 4
    if _mem_available() < pinned + 16 * 2**30:
        pytest.skip(f"host memory: {_mem_available() / 2**30:.0f} GiB available, {pinned / 2**30 + 16:.0f} GiB needed")
    ocfg = oracle.Config(**kw)
    T, V, h, s = cfg.tokens, cfg.vocab, cfg.hidden, cfg.seq
    tok = synth.tokens(T, V)
    lab = synth.labels(T, V)
    with mt.Trainer(cfg) as tr:
        mt.fill_synthetic(cfg, tr.arena, synth, synth.WEIGHT_SEED)
        loss = tr.step(tok, lab)
        x0 = tr.read_checkpoint(0)
        x1 = tr.read_checkpoint(1)
        off, _, _, _ = mt.tensor_offset(cfg, 0, mt.SEC_W, 0)
        E_rows = tr.arena.array[off:off + V * h * 2].view(np.uint16).reshape(V, h)[tok].copy()
        W0 = _f(_bits(mt, cfg, tr.arena, 1, mt.SEC_W))
    expect = math.log(V) + 2e-4 * h
    assert abs(loss - expect) / expect < 0.02, (loss, expect)
    np.testing.assert_array_equal(x0, oracle.bf16_bits_to_float(E_rows, np.float32))

    p = {n: W0[i] for i, n in enumerate(LAYER_NAMES)}
    nh, hd = cfg.n_heads, cfg.head_dim
    rows = np.array([0, 1, 127, 4095, 65536, s - 1])
    cos, sin = om.rope_tables(ocfg, np.float32)
    a, _ = om.rmsnorm(x0, p["attn_norm"], cfg.rms_eps)
    k = om.rope((a @ p["wk"].T).reshape(1, s, nh, hd), cos, sin)[0]
    v = (a @ p["wv"].T).reshape(s, nh, hd)
    q = (a[rows] @ p["wq"].T).reshape(len(rows), nh, hd)
    half = hd // 2
    c, sn = cos[rows][:, None, :], sin[rows][:, None, :]
    q = np.concatenate([q[..., :half] * c - q[..., half:] * sn, q[..., half:] * c + q[..., :half] * sn], axis=-1)
    o = np.empty((len(rows), nh, hd), dtype=np.float32)
    for ri, i in enumerate(rows):
        for n in range(nh):
            sc = (k[: i + 1, n, :] @ q[ri, n, :]) / math.sqrt(hd)
            pr = np.exp(sc - sc.max())
            o[ri, n] = (pr / pr.sum()) @ v[: i + 1, n, :]
    x1_ref = x0[rows] + o.reshape(len(rows), nh * hd) @ p["wo"].T
    bb, _ = om.rmsnorm(x1_ref, p["ffn_norm"], cfg.rms_eps)
    x2_ref = x1_ref + om.swiglu(bb @ p["wg"].T, bb @ p["wu"].T) @ p["wd"].T
    assert _nerr(x1[rows] - x0[rows], x2_ref - x0[rows]) <= 2e-2
