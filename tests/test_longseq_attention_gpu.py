"""Attention kernels at long sequence lengths against the oracle's row-wise attention.

At these lengths the oracle cannot hold an s x s score matrix, so it computes the plain
definition for listed rows (oracle.model.causal_attention_rows and friends, pinned on the
CPU against the full-matrix forms):

* seq 32768, 2 query heads sharing 1 kv head (GQA), oracle in float32: every output row and
  its lse, dq of sampled query rows and dk/dv of sampled key positions, with the oracle's own
  lse and D_i = do_i . o_i for every row;
* seq 131072 (the long-context configuration's length), 1 head, oracle in float64: sampled
  output rows and their lse; dq of sampled rows; dk/dv of sampled key positions,
  teacher-forced with the kernel's lse and o for the rows the oracle does not recompute
  (every row's statistics would take the CPU minutes).

Bars: outputs within 1e-2 and gradients within 2e-2 of the tensor's (sampled) max magnitude,
as in the short-sequence kernel tests; lse within 1e-3 absolute (natural-log units).
"""
import math

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


def _nerr(got, ref):
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))


def _inputs(seed, s, nh, nkv, hd, q_scale, dtype):
    """bf16 q|k|v and do (as numpy copies in `dtype` and GPU tensors); q scaled so the softmax
    rows are peaked enough to move the running maximum."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    qkv = torch.randn(s, (nh + 2 * nkv) * hd, generator=g)
    qkv[:, : nh * hd] *= q_scale
    qkv = qkv.to(torch.bfloat16)
    do = torch.randn(s, nh * hd, generator=g).to(torch.bfloat16)
    return qkv.float().numpy().astype(dtype), qkv.cuda(), do.float().numpy().astype(dtype), do.cuda()


def _split(qkv, nh, nkv, hd):
    q = qkv[:, : nh * hd].reshape(-1, nh, hd)
    k = qkv[:, nh * hd:(nh + nkv) * hd].reshape(-1, nkv, hd)
    v = qkv[:, (nh + nkv) * hd:].reshape(-1, nkv, hd)
    return q, k, v


def _rows(s):
    """Sampled positions: both ends, tile boundaries (64 and 128 rows), and spread interior rows."""
    r = {0, 1, 63, 64, 127, 128, 129, s // 2 - 1, s // 2, s - 129, s - 128, s - 65, s - 64, s - 2, s - 1}
    r |= set(np.random.default_rng(s).integers(0, s, 24).tolist())
    return np.array(sorted(x for x in r if 0 <= x < s))


@pytest.mark.parametrize("s,nh,nkv", [(32768, 2, 1), (131072, 1, 1)])
def test_attention_long_sequence(K, s, nh, nkv):
    hd = 128
    full = s <= 32768
    # every row in float32 at 32768; sampled rows in float64 at 131072
    dt = np.float32 if full else np.float64
    qkv, qkvt, do, dot = _inputs(s + nh, s, nh, nkv, hd, q_scale=2.0, dtype=dt)
    o_t, lse_t = K.attn_fwd(qkvt, 1, s, nh, nkv, hd)
    dqkv = K.attn_bwd(qkvt, o_t, lse_t, dot, 1, s, nh, nkv, hd).float().cpu().numpy()
    o_gpu = o_t.float().cpu().numpy().reshape(s, nh, hd)
    lse_gpu = lse_t.cpu().numpy()[0] * math.log(2.0)  # the kernel keeps log2 of the scaled scores
    q, k, v = _split(qkv, nh, nkv, hd)
    dq_gpu, dk_gpu, dv_gpu = _split(dqkv, nh, nkv, hd)
    do = do.reshape(s, nh, hd)
    rows = _rows(s)
    dk_ref = np.zeros((len(rows), nkv, hd), dtype=dt)
    dv_ref = np.zeros_like(dk_ref)
    for n in range(nh):
        kv = n // (nh // nkv)
        if full:  # every row of the forward
            o_ref, lse_ref = om.causal_attention_all_rows(q[:, n], k[:, kv], v[:, kv], chunk=2048)
            assert _nerr(o_gpu[:, n], o_ref) < 1e-2
            assert np.max(np.abs(lse_gpu[n] - lse_ref)) < 1e-3
            D = np.sum(do[:, n] * o_ref, axis=1)
            lse_b = lse_ref
        else:  # sampled rows of the forward; the backward teacher-forced with the kernel's statistics
            o_ref, lse_ref = om.causal_attention_rows(q[:, n], k[:, kv], v[:, kv], rows)
            assert _nerr(o_gpu[rows, n], o_ref) < 1e-2
            assert np.max(np.abs(lse_gpu[n, rows] - lse_ref)) < 1e-3
            D = np.sum(do[:, n] * o_gpu[:, n].astype(dt), axis=1)
            lse_b = lse_gpu[n].astype(dt)
        dq_ref = om.causal_attention_dq_rows(do[:, n], q[:, n], k[:, kv], v[:, kv], lse_b, D, rows)
        assert _nerr(dq_gpu[rows, n], dq_ref) < 2e-2
        dk_n, dv_n = om.causal_attention_dkv_cols(do[:, n], q[:, n], k[:, kv], v[:, kv], lse_b, D, rows)
        dk_ref[:, kv] += dk_n
        dv_ref[:, kv] += dv_n
    assert _nerr(dk_gpu[rows], dk_ref) < 2e-2
    assert _nerr(dv_gpu[rows], dv_ref) < 2e-2
