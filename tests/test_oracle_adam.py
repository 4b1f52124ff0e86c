"""Pin the oracle's Adam step and bfloat16 rounding to hand-computed values."""
import numpy as np
import pytest

import oracle
from oracle import model as om


def _bits(x):
    return om.float_to_bf16_bits(np.array([x], dtype=np.float64))


def _val(b):
    return float(om.bf16_bits_to_float(b)[0])


def test_bf16_rounding_known_values():
    cases = {
        1.0: 0x3F80, -2.0: 0xC000, 1.0 + 2**-8: 0x3F80,          # tie -> even (down)
        1.0 + 3 * 2**-8: 0x3F82,                                   # tie -> even (up)
        1.0 + 2**-8 + 2**-30: 0x3F81,                              # just above the tie
        0.1: 0x3DCD, -0.02: 0xBCA4, 0.0: 0x0000,
    }
    for x, b in cases.items():
        assert int(_bits(x)[0]) == b, (x, hex(int(_bits(x)[0])), hex(b))
    assert int(_bits(-0.0)[0]) == 0x8000


def test_bf16_rounding_matches_torch_on_float32_inputs():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    # include exact ties
    t = (rng.integers(0, 2**16, 1000).astype(np.uint32) << 16) | 0x8000
    t = t[((t >> 23) & 0xFF) != 0xFF]  # finite values only
    x = np.concatenate([x, t.view(np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(om.float_to_bf16_bits(x.astype(np.float64)), ref)


def _adam(w, g, m, v, t):
    wb, mm, vv = om.adam_update(_bits(w), _bits(g), np.array([m], np.float32), np.array([v], np.float32), t)
    return _val(wb), float(mm[0]), float(vv[0])


def test_adam_first_step_closed_form():
    """w = 0.5, g = bf16(0.1) = 0.10009765625, t = 1: m = 0.1 g, v = 0.001 g^2, mhat = g,
    vhat = g^2, w' = 0.5 - 1e-3 g/(|g| + 1e-8) = 0.49900000001 -> bf16 0.498046875."""
    g = 0.10009765625
    w, m, v = _adam(0.5, 0.1, 0.0, 0.0, 1)
    assert w == 0.498046875
    assert m == np.float32(0.1 * g)
    assert v == np.float32(0.001 * g * g)


def test_adam_second_step_update_lost_to_bf16():
    """Continuing with g = bf16(-0.05) = -0.0500488..., t = 2: m = 0.9 m1 + 0.1 g,
    v = 0.999 v1 + 0.001 g^2; w' = 0.498046875 - 1e-3 mhat/(sqrt(vhat)+eps) ~ 0.49778 -> bf16 0.498046875."""
    w1, m1, v1 = _adam(0.5, 0.1, 0.0, 0.0, 1)
    g = _val(_bits(-0.05))
    w2, m2, v2 = _adam(w1, -0.05, m1, v1, 2)
    m_ref = 0.9 * m1 + 0.1 * g
    v_ref = 0.999 * v1 + 0.001 * g * g
    upd = 1e-3 * (m_ref / (1 - 0.9**2)) / (np.sqrt(v_ref / (1 - 0.999**2)) + 1e-8)
    assert abs((w1 - upd) - 0.4977805) < 1e-6
    assert w2 == 0.498046875
    assert m2 == np.float32(m_ref) and v2 == np.float32(v_ref)


def test_adam_small_weight():
    """w = bf16(-0.02) = -0.02001953125, g = -3e-4, t = 1: w' = w + 1e-3 = -0.01901953 -> bf16 -0.01904296875."""
    w, _, _ = _adam(-0.02, -3e-4, 0.0, 0.0, 1)
    assert w == -0.01904296875


def test_adam_zero_gradient_is_identity():
    w, m, v = _adam(0.375, 0.0, 0.0, 0.0, 1)
    assert (w, m, v) == (0.375, 0.0, 0.0)
    w, m, v = _adam(0.375, 0.0, 0.25, 0.5, 3)
    # m, v decay; w moves by lr * mhat / (sqrt(vhat) + eps) with mhat, vhat from the decayed moments
    assert m == np.float32(0.9 * 0.25) and v == np.float32(0.999 * 0.5)


def test_master_weights_accumulate_what_bf16_rounds_away():
    """Constant gradient g: m_t = g (1 - b1^t) and v_t = g^2 (1 - b2^t), so m_hat = g, v_hat = g^2
    and every step moves the weight by lr g / (|g| + eps). With lr = 1e-4 from w = 0.5 the move is
    far below half a bf16 step under 0.5 (2^-10 = 0.0009765625): without a master copy each step
    rounds back to 0.5 and nothing is ever learned. With an fp32 master the master moves by ~1e-4
    a step; w = bf16(master) stays 0.5 while master > 0.5 - 2^-10 (steps 1..9) and becomes
    0.498046875 (= 255 * 2^-9) at step 10, when master ~ 0.4990."""
    gb = _bits(0.1)
    g = _val(gb)
    step_size = 1e-4 * g / (g + 1e-8)
    w, m, v = _bits(0.5), np.zeros(1, np.float32), np.zeros(1, np.float32)
    for t in range(1, 11):
        w, m, v = om.adam_update(w, gb, m, v, t, lr=1e-4)
        assert _val(w) == 0.5, t
    w, m, v, p = _bits(0.5), np.zeros(1, np.float32), np.zeros(1, np.float32), np.full(1, 0.5, np.float32)
    for t in range(1, 11):
        w, m, v, p = om.adam_update(w, gb, m, v, t, lr=1e-4, master=p)
        assert p.dtype == np.float32
        assert abs(float(p[0]) - (0.5 - t * step_size)) < 1e-6, t
        assert _val(w) == (0.5 if t < 10 else 0.498046875), (t, _val(w))
    # the stored weight is always the bf16 rounding of the stored master
    assert int(w[0]) == int(om.float_to_bf16_bits(p.astype(np.float64))[0])


def test_master_weights_zero_gradient_is_a_fixed_point():
    rng = np.random.default_rng(3)
    p = (rng.standard_normal(1000) * 0.02).astype(np.float32)
    w = om.float_to_bf16_bits(p.astype(np.float64))
    zero = np.zeros(1000, np.uint16)
    m = np.zeros(1000, np.float32)
    w2, m2, v2, p2 = om.adam_update(w, zero, m, m.copy(), 1, master=p)
    np.testing.assert_array_equal(p2, p)
    np.testing.assert_array_equal(w2, w)
    assert not np.any(m2) and not np.any(v2)
