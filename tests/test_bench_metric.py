"""The bench's metric definitions, checked against independent counts (no GPU).

Model FLOPs of a step (6 P_nonemb T + 6 B s^2 h L + 6 T h V, causal attention counted once,
recompute not counted) with P_nonemb taken from the oracle's own list of a decoder block's
tensors, and the per-layer roofline bounded below by each of its resources alone and above by
their sum."""
import numpy as np
import pytest

import bench
import oracle
from oracle import model as om


def _ocfg(kw):
    return oracle.Config(kw["n_layers"], kw["hidden"], kw["n_heads"], kw["n_kv_heads"], kw["ffn"], kw["vocab"],
                         kw["seq"], kw["batch"])


@pytest.mark.parametrize("name", list(bench.CONFIGS))
def test_model_flops_from_the_oracle_parameter_count(name):
    kw = bench.CONFIGS[name]
    cfg = _ocfg(kw)
    p_layer = sum(int(np.prod(shape)) for _, shape in om.block_tensors(cfg, 1))  # a decoder block
    assert bench.layer_params(kw) == p_layer
    T = kw["batch"] * kw["seq"]
    L, h, V, s, B = kw["n_layers"], kw["hidden"], kw["vocab"], kw["seq"], kw["batch"]
    want = 6.0 * p_layer * L * T + 6.0 * B * s * s * h * L + 6.0 * T * h * V
    assert bench.model_flops(kw) == pytest.approx(want, rel=1e-12)


def test_7b_step_flops_value():
    """7B, 8192 tokens: 3.51e14 FLOPs per step (3.18e14 from the 6.476e9 decoder parameters,
    0.26e14 causal attention, 0.06e14 LM head)."""
    f = bench.model_flops(bench.CONFIGS["7b"])
    assert f == pytest.approx(6 * 202383360 * 32 * 8192 + 6 * 2 * 4096**2 * 4096 * 32 + 6 * 8192 * 4096 * 32000)
    assert 3.5e14 < f < 3.52e14


@pytest.mark.parametrize("name", ["1.3b", "7b", "14b", "7b_long"])
@pytest.mark.parametrize("offload", [False, True])
def test_per_layer_roofline_between_single_resource_and_sum(name, offload):
    kw = bench.CONFIGS[name]
    peak, h2d, d2h = 1761.8, 211.0, 193.0
    t = bench.per_layer_roofline_ms(kw, peak, h2d, d2h, offload=offload) / 1e3
    L, h, V, s, B = kw["n_layers"], kw["hidden"], kw["vocab"], kw["seq"], kw["batch"]
    T = B * s
    P = bench.layer_params(kw)
    # one causal-half product (Q K^T, P V, ...) over every head: s^2/2 x hd multiply-adds per head
    unit = B * (s * s / 2) * (kw["n_heads"] * (h // kw["n_heads"])) * 2
    # work: forward (2PT + QK^T, PV), head fwd+bwd (6 T h V), recompute (2PT + QK^T, PV) and
    # backward (4PT + S, dP, dV, dK, dQ)
    flops = L * (2.0 * T * P + 2 * unit) + 6.0 * T * h * V + L * (6.0 * T * P + 7 * unit)
    ck = 4.0 * T * h if offload else 0.0
    h2d_bytes = 2.0 * min(T, V) * h + L * 2.0 * P + 2.0 * (V * h + h) + L * (2.0 * P + ck)
    d2h_bytes = L * ck + 2.0 * (V * h + h) + L * 2.0 * P + 2.0 * min(2 * T, V) * h
    parts = (flops / (peak * 1e12), h2d_bytes / (h2d * 1e9), d2h_bytes / (d2h * 1e9))
    assert t >= max(parts) * (1 - 1e-9)
    assert t <= sum(parts) * (1 + 1e-9)
