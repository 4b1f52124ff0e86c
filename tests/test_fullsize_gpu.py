"""Parity at the benchmark configurations' full sizes, in the launch configuration bench.py times.

A whole-model oracle step at these sizes would take the CPU hours, so the oracle is
teacher-forced, layer by layer, from the GPU step's own layer-boundary checkpoints
(mt_read_checkpoint) and upstream gradients (mt_capture_input_grad):

* x_0 equals the embedding rows of the tokens exactly;
* the loss, the head's gradients (final norm, LM head) and dL/dx_L, recomputed by the oracle
  from the GPU's final hidden state x_L;
* decoder layers 0, L/2 and L-1: the forward x_l -> x_{l+1} from the GPU's x_l, and the
  backward from the GPU's dL/dx_{l+1}: all nine weight gradients and dL/dx_l;
* the embedding gradient rows, the ordered scatter of the GPU's dL/dx_0;
* the initial loss against its closed form ln V + 2e-4 h;
* 1.3B runs the configuration's three streamed steps with the host Adam between them: after
  every step the oracle's Adam applied to that step's gradients and moments gives the
  product's updated W, m and v, and every step's loss is the oracle's head loss; the layer
  checks above run on the third step, where the Adam state has fed back twice.

Bars as everywhere: loss 1e-3 relative, tensors 2e-2 of their max magnitude (the teacher-forced
Adam 2.5e-3, as in the small-config test). The oracle runs in float32 here (its float32
instantiation is pinned to float64 on the CPU). Host memory is checked before each
configuration; one that does not fit is skipped with the reason.
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


def _teacher_forced_layer(ocfg, l, x_in, x_out, dy, W, G, dx_gpu, cos, sin):
    """Layer l by the oracle from the GPU's input x_l and upstream gradient dL/dx_{l+1}."""
    p = {n: W[i] for i, n in enumerate(LAYER_NAMES)}
    ref_out, cache = om.layer_forward(x_in, p, ocfg, cos, sin)
    errs = {"fwd": _nerr(x_out - x_in, ref_out - x_in)}
    dx, g = om.layer_backward(dy, cache, p, ocfg, cos, sin)
    errs["dx"] = _nerr(dx_gpu, dx)
    for i, n in enumerate(LAYER_NAMES):
        errs[n] = _nerr(G[i], g[n])
    bad = {k: v for k, v in errs.items() if v > 2e-2}
    assert not bad, (l, bad)
    return errs


def _adam_teacher_forced(ocfg, before, after, step):
    """The oracle's Adam on the arena as the step left it (W, G, M, V) against the product's.

    Both sides round the same update to bf16, the product from fp32 and the oracle from float64,
    so an updated weight may differ by one bf16 step where the exact result lies next to a
    rounding boundary: every weight must be within one bf16 step of the oracle's (a step is
    2^-8 to 2^-7 of the value; 2^-7 of the larger of the two) plus the fp32 rounding of the
    subtraction where the old weight and the step nearly cancel, m and v within fp32 rounding
    (1e-5 of the tensor's max), and each tensor within the stated 2e-2 bar. Returns (worst
    normalised weight error, weights one step apart)."""
    B = oracle.unpack_arena(ocfg, before, "W"), oracle.unpack_arena(ocfg, before, "G")
    M0, V0 = oracle.unpack_arena(ocfg, before, "M"), oracle.unpack_arena(ocfg, before, "V")
    W1, M1, V1 = (oracle.unpack_arena(ocfg, after, sec) for sec in "WMV")
    worst, one_step = 0.0, 0
    for b in range(len(W1)):
        for name in W1[b]:
            w, m, v = oracle.adam_update(B[0][b][name], B[1][b][name], M0[b][name], V0[b][name], step)
            ew = oracle.bf16_bits_to_float(w)
            gw = oracle.bf16_bits_to_float(W1[b][name])
            w0 = oracle.bf16_bits_to_float(B[0][b][name])
            d = np.abs(gw - ew)
            # one bf16 step of the result, plus the fp32 rounding of w - step where the two nearly
            # cancel (Adam's first steps are about lr in size, like many small weights)
            ok = bool(np.all(d <= 2.0 ** -7 * np.maximum(np.abs(ew), np.abs(gw)) + 2.0 ** -20 * (np.abs(w0) + 1e-3)))
            e = _nerr(gw, ew)
            em, ev = _nerr(M1[b][name], m), _nerr(V1[b][name], v)
            assert ok and e <= 2e-2 and em <= 1e-5 and ev <= 1e-5, (step, b, name, ok, e, em, ev)
            worst = max(worst, e)
            one_step += int(np.count_nonzero(d))
    return worst, one_step


@pytest.mark.parametrize("name", list(CFGS))
def test_fullsize_teacher_forced(mt, name):
    kw = dict(CFGS[name])
    steps = 3 if name == "1.3b" else 1
    copies = 3 if steps > 1 else 1  # the arena and, for the Adam checks, two copies of it
    need = mt.arena_bytes(mt.ModelConfig(**kw)) * copies + 12 * 2**30
    while _mem_available() < need and kw["n_layers"] > 4:
        # a host that cannot hold the whole arena runs the same layer shapes with fewer layers
        # (every checked layer, the head and the embedding have the configuration's sizes)
        kw["n_layers"] -= 4
        need = mt.arena_bytes(mt.ModelConfig(**kw)) * copies + 12 * 2**30
    if _mem_available() < need:
        pytest.skip(f"host memory: {_mem_available() / 2**30:.0f} GiB available, {need / 2**30:.0f} GiB needed")
    if kw["n_layers"] != CFGS[name]["n_layers"]:
        print(f"{name}: host memory holds {kw['n_layers']} of {CFGS[name]['n_layers']} layers")
    cfg = mt.ModelConfig(**kw)
    ocfg = oracle.Config(**kw)
    L, T, V, h = cfg.n_layers, cfg.tokens, cfg.vocab, cfg.hidden
    tok = synth.tokens(T, V)
    lab = synth.labels(T, V)
    dt = np.float32
    layers = sorted({0, L // 2, L - 1})
    ph_head = None
    losses, head_losses, adam_report = [], [], []
    # run the steps, copy what the oracle needs (bf16 bit patterns, checkpoints, boundary
    # gradients), then free the pinned arena before the oracle's large arrays
    with mt.Trainer(cfg) as tr:
        mt.fill_synthetic(cfg, tr.arena, synth, synth.WEIGHT_SEED)
        caps = {l: tr.capture_input_grad(l) for l in sorted({L} | set(layers) | {l + 1 for l in layers})}
        for step in range(1, steps + 1):
            losses.append(tr.step(tok, lab))
            xL = tr.read_checkpoint(L)
            Whead = _f(_bits(mt, cfg, tr.arena, L + 1, mt.SEC_W))
            ph_head = {"final_norm": Whead[0], "w_head": Whead[1]}
            head_losses.append(om.head_forward_backward(xL.astype(dt), ph_head, lab, ocfg)[0])
            if step < steps:
                before = tr.arena.array.copy()
                tr.adam(step)
                after = tr.arena.array.copy()  # a copy: an assertion's report must not read freed memory
                adam_report.append(_adam_teacher_forced(ocfg, before, after, step))
                del before, after
        x = {l: tr.read_checkpoint(l) for l in sorted(set(layers) | {l + 1 for l in layers})}
        dxs = {l: caps[l].copy() for l in caps}
        del caps  # views of page-locked buffers that close() frees
        off, _, _, _ = mt.tensor_offset(cfg, 0, mt.SEC_W, 0)
        E_rows = tr.arena.array[off:off + V * h * 2].view(np.uint16).reshape(V, h)[tok].copy()
        uniq = np.unique(tok)
        off, _, _, _ = mt.tensor_offset(cfg, 0, mt.SEC_G, 0)
        GE_rows = tr.arena.array[off:off + V * h * 2].view(np.uint16).reshape(V, h)[uniq].copy()
        Wl = {l: _f(_bits(mt, cfg, tr.arena, l + 1, mt.SEC_W)) for l in layers}
        Gl = {l: _f(_bits(mt, cfg, tr.arena, l + 1, mt.SEC_G)) for l in layers}
        Ghead = _f(_bits(mt, cfg, tr.arena, L + 1, mt.SEC_G))

    for a, b in zip(losses, head_losses):
        assert abs(a - b) <= 1e-3 * abs(b), (losses, head_losses)
    if steps == 1:
        # the initial loss against its closed form (unit gains, N(0, 0.02^2) head)
        expect = math.log(V) + 2e-4 * h
        assert abs(losses[0] - expect) / expect < 0.02, (losses[0], expect)
    else:
        assert losses[-1] < losses[0]  # the same batch three times: the loss goes down
    # embedding gather: exact
    np.testing.assert_array_equal(x[0], oracle.bf16_bits_to_float(E_rows, np.float32))

    # head, teacher-forced from the GPU's x_L (last step)
    ref_loss, dxL, gh, _ = om.head_forward_backward(xL.astype(dt), ph_head, lab, ocfg)
    assert _nerr(Ghead[0], gh["final_norm"]) <= 2e-2
    assert _nerr(Ghead[1], gh["w_head"]) <= 2e-2
    assert _nerr(dxs[L], dxL) <= 2e-2
    del gh

    cos, sin = om.rope_tables(ocfg, dt)
    report = {}
    for l in layers:
        report[l] = _teacher_forced_layer(ocfg, l, x[l].astype(dt), x[l + 1], dxs[l + 1], Wl[l], Gl[l], dxs[l],
                                          cos, sin)
    # embedding gradient: the ordered scatter of dL/dx_0, on the rows this batch touched
    dE = om.embedding_backward(dxs[0], tok, V)[uniq]
    assert _nerr(oracle.bf16_bits_to_float(GE_rows, np.float32), dE) <= 2e-2
    print(f"{name}: worst normalised error per checked layer", {l: max(v.values()) for l, v in report.items()},
          "teacher-forced Adam (worst weight error, weights one bf16 step from the oracle's):", adam_report)


@pytest.mark.parametrize("seq", [131072, 262144])
def test_fullsize_long_context_sampled_rows(mt, seq):
    """7B shape at seq 131072 (checkpoints offloaded to pinned host memory) and 262144.

    The oracle cannot hold 131072 x 131072 attention matrices, so layer 0 is recomputed on
    sampled query positions only: RMSNorm, q/k/v, RoPE and causal attention over every earlier
    key of those rows, the output projection, the FFN. Its x_1 rows are compared with the
    GPU's checkpoint x_1 (read back from the host copy), plus the exact embedding gather, the
    closed-form initial loss, and the embedding gradient (the ordered scatter of the step's
    dL/dx_0 over all 131072 positions). The attention backward at this length is checked at
    kernel level against the oracle's row-wise attention (test_longseq_attention_gpu.py).
    """
    kw = dict(n_layers=32, hidden=4096, n_heads=32, n_kv_heads=32, ffn=11008, vocab=32000, seq=seq, batch=1)
    # 131072: checkpoints offloaded to pinned host memory; 262144: checkpoints in HBM (the host
    # could not hold 32 x 4.3 GB of them next to the arena), LM head in chunks
    offload = seq == 131072
    cfg = mt.ModelConfig(**kw, flags=mt.FLAG_OFFLOAD_CKPT if offload else 0)
    pinned = mt.arena_bytes(cfg) + (cfg.n_layers if offload else 1) * cfg.tokens * cfg.hidden * 4
    if _mem_available() < pinned + 24 * 2**30:
        pytest.skip(f"host memory: {_mem_available() / 2**30:.0f} GiB available, {pinned / 2**30 + 24:.0f} GiB needed")
    torch.cuda.empty_cache()  # earlier tests' workspaces stay cached by the allocator otherwise
    if torch.cuda.mem_get_info()[0] < mt.workspace_bytes(cfg) + 4 * 2**30:
        pytest.skip(f"device memory: {torch.cuda.mem_get_info()[0] / 2**30:.0f} GiB free, "
                    f"{mt.workspace_bytes(cfg) / 2**30 + 4:.0f} GiB needed")
    ocfg = oracle.Config(**kw)
    T, V, h, s = cfg.tokens, cfg.vocab, cfg.hidden, cfg.seq
    tok = synth.tokens(T, V)
    lab = synth.labels(T, V)
    with mt.Trainer(cfg) as tr:
        mt.fill_synthetic(cfg, tr.arena, synth, synth.WEIGHT_SEED)
        cap0 = tr.capture_input_grad(0)
        loss = tr.step(tok, lab)
        x0 = tr.read_checkpoint(0)
        x1 = tr.read_checkpoint(1)
        dx0 = cap0.copy()
        del cap0  # a view of a page-locked buffer that close() frees
        off, _, _, _ = mt.tensor_offset(cfg, 0, mt.SEC_W, 0)
        E_rows = tr.arena.array[off:off + V * h * 2].view(np.uint16).reshape(V, h)[tok].copy()
        uniq = np.unique(tok)
        off, _, _, _ = mt.tensor_offset(cfg, 0, mt.SEC_G, 0)
        GE_rows = tr.arena.array[off:off + V * h * 2].view(np.uint16).reshape(V, h)[uniq].copy()
        W0 = _f(_bits(mt, cfg, tr.arena, 1, mt.SEC_W))
    # the embedding backward at this length: the ordered scatter of the step's own dL/dx_0
    # (131072 positions into the rows the batch touched), written straight into the arena
    dE = om.embedding_backward(dx0, tok, V)[uniq]
    assert _nerr(oracle.bf16_bits_to_float(GE_rows, np.float32), dE) <= 2e-2
    assert np.all(np.isfinite(dx0))
    del dx0, dE
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


def test_fullsize_schedules_bitwise_1p3b(mt):
    """1.3B, two steps with the host Adam after each: the streamed schedule (four weight pieces
    per layer, each with its own event, two layer buffers) leaves the whole arena bit-identical
    to the resident schedule and to the streamed schedule with checkpoints offloaded."""
    kw = CFGS["1.3b"]
    cfg = mt.ModelConfig(**kw)
    T = cfg.tokens
    need = 2 * mt.arena_bytes(cfg) + cfg.n_layers * T * cfg.hidden * 4 + 12 * 2**30
    if _mem_available() < need:
        pytest.skip(f"host memory: {_mem_available() / 2**30:.0f} GiB available, {need / 2**30:.0f} GiB needed")
    tok = synth.tokens(T, cfg.vocab)
    lab = synth.labels(T, cfg.vocab)

    def run(flags):
        c = mt.ModelConfig(**kw, flags=flags)
        with mt.Trainer(c) as tr:
            mt.fill_synthetic(c, tr.arena, synth, synth.WEIGHT_SEED)
            losses = []
            for step in (1, 2):
                losses.append(tr.step(tok, lab))
                tr.adam(step)
            return losses, tr.arena.array.copy()

    ref_losses, ref = run(mt.FLAG_RESIDENT)
    for flags in (0, mt.FLAG_OFFLOAD_CKPT):
        losses, arena = run(flags)
        assert losses == ref_losses, (flags, losses, ref_losses)
        assert np.array_equal(arena, ref), flags
        del arena
