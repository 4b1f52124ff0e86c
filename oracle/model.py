"""Oracle model: layout, unpacking, forward, backward and Adam, written out plainly.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources, by page and section:
  * chatpaper abstract ("MegaTrain: Full Precision Training of 100B+ Parameter
    Large Language Models on a Single GPU", Abstract): per layer, parameters
    stream in and gradients stream out; parameters and optimizer states live
    in host memory.
  * chestersoft digest ("MegaTrain", Methodik, "Layer-Contiguous Tiling"):
    each layer's state (BF16 weights, BF16 gradients, FP32 Adam moments) is
    packed into a contiguous 4 KB-aligned block; the optimizer step runs on
    the CPU.
  * ecosistemastartup article ("MegaTrain: entrena LLMs de 100B+ en una sola
    GPU", Innovaciones 1): the GPU receives a layer's weights, runs forward
    and backward, and returns the gradients.
The pages give no model equations. The model is the Llama-style decoder of
the benchmark configurations: RMSNorm, rotate-half RoPE, causal grouped-query
attention, SwiGLU, untied embedding and LM head, no biases, mean token
cross-entropy. Readings taken where the pages are silent:
  R1 stored W and G are bfloat16, Adam m and v float32, no float32 master copy.
  R2 plain bias-corrected Adam, no weight decay, applied to every tensor.
  R3 G is overwritten by each step.
  R4 embedding block E first, decoder blocks, then head block H (final norm
     gain and LM head).
  R5 RMSNorm eps 1e-5, gains initialised to 1, RoPE theta 1e4, angle
     computed in float64, head_dim = hidden / heads.
  R6 loss = mean over all batch*seq positions of lse - z[label].
  R8 block layout: sections W, G, M, V; every section and every tensor starts
     on a 4096-byte boundary relative to the 4096-aligned arena; tensor order
     attn_norm, wq, wk, wv, wo, ffn_norm, wg, wu, wd (E: emb; H: final_norm,
     w_head); matrices row-major [out, in].
  R18 optional float32 master weights (the digest's "full precision" taken the
     other way from R1): a fifth section P (float32, same tensor order) after V;
     Adam moves P, computed in float64 and stored as float32, and W becomes the
     bfloat16 (nearest even) of the stored P.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

ALIGN = 4096


# ----------------------------------------------------------------------------
# configuration
# ----------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Config:
    n_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    ffn: int
    vocab: int
    seq: int
    batch: int
    rms_eps: float = 1e-5
    rope_theta: float = 10000.0
    fp32_master: bool = False  # R18: a float32 master section P in every block

    @property
    def head_dim(self) -> int:
        return self.hidden // self.n_heads

    @property
    def tokens(self) -> int:
        return self.batch * self.seq


# ----------------------------------------------------------------------------
# bfloat16 <-> float (round to nearest even), written from the format's definition
# ----------------------------------------------------------------------------
def bf16_bits_to_float(bits: np.ndarray, dtype=np.float64) -> np.ndarray:
    """bfloat16 is the upper half of an IEEE binary32 word."""
    u32 = bits.astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(dtype)


def float_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bfloat16 (8 significant bits), ties to even.

    With x = m * 2^e, 0.5 <= |m| < 1 (frexp), the bfloat16 quantum is
    2^(max(e, -125) - 8) (the floor gives the subnormal spacing 2^-133).
    ``numpy.rint`` rounds half to even. The rounded value is exact in float32,
    whose upper 16 bits are the bfloat16 pattern. Float64 input is rounded
    once, directly.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    q = np.ldexp(1.0, np.maximum(e, -125) - 8)
    r = np.rint(x / q) * q
    return (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# ----------------------------------------------------------------------------
# packed-block layout (reading R8), computed from the written rule
# ----------------------------------------------------------------------------
def _round_up(n: int, a: int = ALIGN) -> int:
    return (n + a - 1) // a * a


def block_tensors(cfg: Config, block: int):
    """(name, shape) of the tensors of block ``block`` in storage order."""
    h, f, V = cfg.hidden, cfg.ffn, cfg.vocab
    qd = cfg.n_heads * cfg.head_dim
    kvd = cfg.n_kv_heads * cfg.head_dim
    if block == 0:
        return [("emb", (V, h))]
    if block == cfg.n_layers + 1:
        return [("final_norm", (h,)), ("w_head", (V, h))]
    return [
        ("attn_norm", (h,)),
        ("wq", (qd, h)),
        ("wk", (kvd, h)),
        ("wv", (kvd, h)),
        ("wo", (h, qd)),
        ("ffn_norm", (h,)),
        ("wg", (f, h)),
        ("wu", (f, h)),
        ("wd", (h, f)),
    ]


def layout(cfg: Config):
    """Byte offsets of every block, section and tensor in the host arena.

    Returns a dict with ``total`` and ``blocks``: a list, one entry per block,
    each {"offset", "bytes", "sections": {sec: {"offset", "bytes",
    "tensors": {name: offset}}}} with offsets relative to the arena base.
    Sections W, G hold bfloat16 (2 bytes/element), M, V float32 (4 bytes), and with
    ``cfg.fp32_master`` a fifth section P, float32 (R18).
    """
    sections = [("W", 2), ("G", 2), ("M", 4), ("V", 4)] + ([("P", 4)] if cfg.fp32_master else [])
    blocks = []
    off = 0
    for b in range(cfg.n_layers + 2):
        tens = block_tensors(cfg, b)
        bstart = off
        secs = {}
        for sec, esz in sections:
            sstart = off
            toffs = {}
            for name, shape in tens:
                toffs[name] = off
                off = _round_up(off + int(np.prod(shape)) * esz)
            secs[sec] = {"offset": sstart, "bytes": off - sstart, "tensors": toffs}
        blocks.append({"offset": bstart, "bytes": off - bstart, "sections": secs})
    return {"total": off, "blocks": blocks}


def init_params(cfg: Config, synth, seed: int):
    """Initial weights as bfloat16 bit patterns, from the shared generator.

    Gains are 1.0; every matrix and the embedding are N(0, 0.02^2).
    """
    out = []
    for b in range(cfg.n_layers + 2):
        d = {}
        for ti, (name, shape) in enumerate(block_tensors(cfg, b)):
            n = int(np.prod(shape))
            if len(shape) == 1:
                d[name] = synth.const_bf16(n, 1.0).reshape(shape)
            else:
                d[name] = synth.normal_bf16(n, seed, synth.weight_stream(b, ti)).reshape(shape)
        out.append(d)
    return out


def pack_arena(cfg: Config, weights_bits, lay=None) -> np.ndarray:
    """Bytes of a freshly initialised arena: W = weights, G = M = V = 0 (and P = W as float32)."""
    lay = lay or layout(cfg)
    arena = np.zeros(lay["total"], dtype=np.uint8)
    for b, blk in enumerate(lay["blocks"]):
        for name, _ in block_tensors(cfg, b):
            o = blk["sections"]["W"]["tensors"][name]
            raw = np.ascontiguousarray(weights_bits[b][name]).view(np.uint8).ravel()
            arena[o:o + raw.size] = raw
            if cfg.fp32_master:
                o = blk["sections"]["P"]["tensors"][name]
                pm = bf16_bits_to_float(np.ascontiguousarray(weights_bits[b][name])).astype(np.float32)
                arena[o:o + pm.nbytes] = pm.view(np.uint8).ravel()
    return arena


def unpack_arena(cfg: Config, arena: np.ndarray, section: str, lay=None):
    """Per block, a dict name -> array of section ``section`` (uint16 bits for W/G, float32 for M/V/P)."""
    lay = lay or layout(cfg)
    dt = np.uint16 if section in ("W", "G") else np.float32
    esz = 2 if section in ("W", "G") else 4
    out = []
    for b, blk in enumerate(lay["blocks"]):
        d = {}
        for name, shape in block_tensors(cfg, b):
            o = blk["sections"][section]["tensors"][name]
            n = int(np.prod(shape))
            d[name] = arena[o:o + n * esz].view(dt).reshape(shape)
        out.append(d)
    return out


# ----------------------------------------------------------------------------
# model pieces
# ----------------------------------------------------------------------------
def rmsnorm(x, gamma, eps):
    """y = x / sqrt(mean(x^2) + eps) * gamma; also returns the per-row 1/rms."""
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return x * r * gamma, r


def rmsnorm_backward(dy, x, gamma, r):
    """Gradient of rmsnorm w.r.t. x and gamma (chain rule through r)."""
    xhat = x * r
    dgamma = np.sum(dy * xhat, axis=0)
    dxhat = dy * gamma
    dx = r * (dxhat - xhat * np.mean(dxhat * xhat, axis=-1, keepdims=True))
    return dx, dgamma


def rope_tables(cfg: Config, dtype):
    """cos and sin of angle pos * theta^(-2i/hd), i < hd/2, computed in float64."""
    hd = cfg.head_dim
    i = np.arange(hd // 2, dtype=np.float64)
    inv_freq = cfg.rope_theta ** (-2.0 * i / hd)
    pos = np.arange(cfg.seq, dtype=np.float64)
    ang = pos[:, None] * inv_freq[None, :]
    return np.cos(ang).astype(dtype), np.sin(ang).astype(dtype)


def rope(x, cos, sin):
    """Rotate-half RoPE on x[B, s, heads, hd]: pairs (i, i + hd/2) rotate by the angle."""
    half = x.shape[-1] // 2
    x1, x2 = x[..., :half], x[..., half:]
    c = cos[None, :, None, :]
    s = sin[None, :, None, :]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def rope_backward(dy, cos, sin):
    """Transpose of the rotation, i.e. rotation by the negative angle."""
    half = dy.shape[-1] // 2
    d1, d2 = dy[..., :half], dy[..., half:]
    c = cos[None, :, None, :]
    s = sin[None, :, None, :]
    return np.concatenate([d1 * c + d2 * s, d2 * c - d1 * s], axis=-1)


def causal_attention(q, k, v):
    """o[b,i,n] = sum_j softmax_j(q_i . k_j / sqrt(hd), j <= i) v_j, kv head = n // (nh/nkv).

    q [B, s, nh, hd], k and v [B, s, nkv, hd]. Returns o and the probabilities P
    [B, nh, s, s] (kept for the backward pass).
    """
    B, s, nh, hd = q.shape
    nkv = k.shape[2]
    group = nh // nkv
    scale = 1.0 / math.sqrt(hd)
    mask = np.triu(np.ones((s, s), dtype=bool), k=1)
    o = np.empty_like(q)
    P = np.empty((B, nh, s, s), dtype=q.dtype)
    for b in range(B):
        for n in range(nh):
            kv = n // group
            S = (q[b, :, n, :] @ k[b, :, kv, :].T) * scale
            S = np.where(mask, -np.inf, S)
            S = S - S.max(axis=1, keepdims=True)
            E = np.exp(S)
            Pn = E / E.sum(axis=1, keepdims=True)
            P[b, n] = Pn
            o[b, :, n, :] = Pn @ v[b, :, kv, :]
    return o, P


def causal_attention_backward(do, q, k, v, P):
    """Gradients of causal_attention w.r.t. q, k, v (GQA: k, v sum over their query heads)."""
    B, s, nh, hd = q.shape
    nkv = k.shape[2]
    group = nh // nkv
    scale = 1.0 / math.sqrt(hd)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for n in range(nh):
            kv = n // group
            Pn = P[b, n]
            don = do[b, :, n, :]
            dv[b, :, kv, :] += Pn.T @ don
            dP = don @ v[b, :, kv, :].T
            dS = Pn * (dP - np.sum(dP * Pn, axis=1, keepdims=True))
            dq[b, :, n, :] = (dS @ k[b, :, kv, :]) * scale
            dk[b, :, kv, :] += (dS.T @ q[b, :, n, :]) * scale
    return dq, dk, dv


def causal_attention_rows(q, k, v, rows):
    """Causal attention of one head for the listed query rows only, by the same definition as
    causal_attention: for row i, S_j = q_i . k_j / sqrt(hd) over keys j <= i, P = softmax(S),
    o_i = sum_j P_j v_j. Also returns lse_i = log sum_j exp(S_j) (natural log, scaled scores).
    q, k, v: [s, hd] of one (batch, head) pair; rows: query positions. Each listed row is
    computed on its own (the rows are stacked only to use one matrix product for them), so the
    length s is not bounded by an s x s matrix.
    """
    rows = np.asarray(rows)
    hd = q.shape[1]
    scale = 1.0 / math.sqrt(hd)
    n = int(rows.max()) + 1
    S = (q[rows] @ k[:n].T) * scale
    S = np.where(np.arange(n)[None, :] > rows[:, None], -np.inf, S)
    smax = S.max(axis=1, keepdims=True)
    E = np.exp(S - smax)
    z = E.sum(axis=1, keepdims=True)
    o = (E / z) @ v[:n]
    return o, (smax + np.log(z))[:, 0]


def causal_attention_all_rows(q, k, v, chunk=1024):
    """o [s, hd] and lse [s] of one head for every query row, causal_attention_rows applied to
    consecutive chunks of rows (rows are independent of one another)."""
    s = q.shape[0]
    o = np.empty_like(q)
    lse = np.empty(s, dtype=q.dtype)
    for r0 in range(0, s, chunk):
        rows = np.arange(r0, min(s, r0 + chunk))
        o[rows], lse[rows] = causal_attention_rows(q, k, v, rows)
    return o, lse


def causal_attention_backward_rows(do, q, k, v, o, lse, chunk=1024):
    """dq, dk, dv of one head (causal_attention_backward for one (batch, head) pair) from the
    forward's o and lse, without an s x s matrix: P_ij = exp(S_ij - lse_i) for j <= i,
    dP_ij = do_i . v_j, D_i = sum_j P_ij dP_ij = do_i . o_i, dS_ij = P_ij (dP_ij - D_i);
    dq_i = sum_j dS_ij k_j / sqrt(hd), dk_j = sum_i dS_ij q_i / sqrt(hd), dv_j = sum_i P_ij do_i.
    Query rows are taken in consecutive chunks; the sums over i for dk and dv are accumulated
    chunk after chunk (the same sum, summed in row order)."""
    s, hd = q.shape
    scale = 1.0 / math.sqrt(hd)
    D = np.sum(do * o, axis=1)
    dq = np.empty_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for r0 in range(0, s, chunk):
        rows = np.arange(r0, min(s, r0 + chunk))
        n = int(rows[-1]) + 1
        S = (q[rows] @ k[:n].T) * scale
        P = np.where(np.arange(n)[None, :] > rows[:, None], 0.0, np.exp(S - lse[rows][:, None]))
        dP = do[rows] @ v[:n].T
        dS = P * (dP - D[rows][:, None])
        dq[rows] = (dS @ k[:n]) * scale
        dk[:n] += (dS.T @ q[rows]) * scale
        dv[:n] += P.T @ do[rows]
    return dq, dk, dv


def causal_attention_dq_rows(do, q, k, v, lse, D, rows):
    """dq of one head for the listed query rows only (the definition in
    causal_attention_backward_rows, row by row): needs that row's lse_i and D_i = do_i . o_i."""
    rows = np.asarray(rows)
    hd = q.shape[1]
    scale = 1.0 / math.sqrt(hd)
    n = int(rows.max()) + 1
    S = (q[rows] @ k[:n].T) * scale
    P = np.where(np.arange(n)[None, :] > rows[:, None], 0.0, np.exp(S - lse[rows][:, None]))
    dS = P * (do[rows] @ v[:n].T - D[rows][:, None])
    return (dS @ k[:n]) * scale


def causal_attention_dkv_cols(do, q, k, v, lse, D, cols):
    """dk and dv of one head for the listed key positions only: for key j, over the query rows
    i >= j that see it, P_ij = exp(q_i . k_j / sqrt(hd) - lse_i), dS_ij = P_ij (do_i . v_j - D_i),
    dk_j = sum_i dS_ij q_i / sqrt(hd), dv_j = sum_i P_ij do_i. lse and D cover every row."""
    cols = np.asarray(cols)
    hd = q.shape[1]
    scale = 1.0 / math.sqrt(hd)
    dk = np.empty((len(cols), hd), dtype=q.dtype)
    dv = np.empty((len(cols), hd), dtype=q.dtype)
    for c, j in enumerate(cols):
        P = np.exp((q[j:] @ k[j]) * scale - lse[j:])
        dS = P * (do[j:] @ v[j] - D[j:])
        dk[c] = (dS @ q[j:]) * scale
        dv[c] = P @ do[j:]
    return dk, dv


def silu(z):
    return z / (1.0 + np.exp(-z))


def swiglu(g, u):
    """SwiGLU activation silu(g) * u."""
    return silu(g) * u


def swiglu_backward(dact, g, u):
    """Gradients of silu(g) * u: silu'(g) = sig(g) (1 + g (1 - sig(g)))."""
    sig = 1.0 / (1.0 + np.exp(-g))
    return dact * u * sig * (1.0 + g * (1.0 - sig)), dact * g * sig


def cross_entropy(z, labels):
    """Per-row loss lse(z_t) - z_t[label_t] and the gradient of their mean, (softmax - onehot) / T."""
    T = z.shape[0]
    zmax = z.max(axis=1, keepdims=True)
    lse = zmax[:, 0] + np.log(np.sum(np.exp(z - zmax), axis=1))
    rows = lse - z[np.arange(T), labels]
    dz = np.exp(z - lse[:, None])
    dz[np.arange(T), labels] -= 1.0
    dz /= T
    return rows, dz


def embedding_backward(dx, tokens, vocab):
    """dE[v] = sum of dx[t] over positions t (ascending) holding token v."""
    demb = np.zeros((vocab, dx.shape[1]), dtype=dx.dtype)
    for t in range(tokens.size):
        demb[tokens[t]] += dx[t]
    return demb


def layer_forward(x, p, cfg: Config, cos, sin):
    """One decoder layer on the residual stream x [T, h]; returns x_out and a cache."""
    B, s = cfg.batch, cfg.seq
    nh, nkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    a, r1 = rmsnorm(x, p["attn_norm"], cfg.rms_eps)
    q = (a @ p["wq"].T).reshape(B, s, nh, hd)
    k = (a @ p["wk"].T).reshape(B, s, nkv, hd)
    v = (a @ p["wv"].T).reshape(B, s, nkv, hd)
    qr, kr = rope(q, cos, sin), rope(k, cos, sin)
    o, P = causal_attention(qr, kr, v)
    of = o.reshape(B * s, nh * hd)
    x1 = x + of @ p["wo"].T
    bb, r2 = rmsnorm(x1, p["ffn_norm"], cfg.rms_eps)
    g = bb @ p["wg"].T
    u = bb @ p["wu"].T
    act = swiglu(g, u)
    x2 = x1 + act @ p["wd"].T
    cache = dict(x=x, a=a, r1=r1, qr=qr, kr=kr, v=v, P=P, of=of, x1=x1, bb=bb, r2=r2, g=g, u=u, act=act)
    return x2, cache


def layer_backward(dx2, c, p, cfg: Config, cos, sin):
    """Chain rule back through layer_forward; returns dx and the parameter gradients."""
    B, s = cfg.batch, cfg.seq
    nh, nkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    grads = {}
    # x2 = x1 + act Wd^T
    grads["wd"] = dx2.T @ c["act"]
    dact = dx2 @ p["wd"]
    dg, du = swiglu_backward(dact, c["g"], c["u"])
    grads["wg"] = dg.T @ c["bb"]
    grads["wu"] = du.T @ c["bb"]
    dbb = dg @ p["wg"] + du @ p["wu"]
    dx1_norm, grads["ffn_norm"] = rmsnorm_backward(dbb, c["x1"], p["ffn_norm"], c["r2"])
    dx1 = dx2 + dx1_norm
    # x1 = x + o Wo^T
    grads["wo"] = dx1.T @ c["of"]
    do = (dx1 @ p["wo"]).reshape(B, s, nh, hd)
    dqr, dkr, dv = causal_attention_backward(do, c["qr"], c["kr"], c["v"], c["P"])
    dq = rope_backward(dqr, cos, sin).reshape(B * s, nh * hd)
    dk = rope_backward(dkr, cos, sin).reshape(B * s, nkv * hd)
    dv = dv.reshape(B * s, nkv * hd)
    a = c["a"]
    grads["wq"] = dq.T @ a
    grads["wk"] = dk.T @ a
    grads["wv"] = dv.T @ a
    da = dq @ p["wq"] + dk @ p["wk"] + dv @ p["wv"]
    dx_norm, grads["attn_norm"] = rmsnorm_backward(da, c["x"], p["attn_norm"], c["r1"])
    return dx1 + dx_norm, grads


def head_forward_backward(x, p, labels, cfg: Config):
    """Final RMSNorm, LM head, mean cross-entropy; returns loss, dx and the head gradients."""
    T = x.shape[0]
    y, r = rmsnorm(x, p["final_norm"], cfg.rms_eps)
    z = y @ p["w_head"].T
    rows, dz = cross_entropy(z, labels)
    loss = np.mean(rows)
    grads = {"w_head": dz.T @ y}
    dy = dz @ p["w_head"]
    dx, grads["final_norm"] = rmsnorm_backward(dy, x, p["final_norm"], r)
    return loss, dx, grads, z


def loss_only(cfg: Config, weights, tokens, labels, dtype=np.float64):
    """Forward pass only: the mean cross-entropy for float (or bfloat16-bit) weights."""
    W = [{k: (bf16_bits_to_float(v, dtype) if v.dtype == np.uint16 else v.astype(dtype))
          for k, v in blk.items()} for blk in weights]
    tokens = np.asarray(tokens).reshape(-1)
    labels = np.asarray(labels).reshape(-1)
    cos, sin = rope_tables(cfg, dtype)
    x = W[0]["emb"][tokens]
    for l in range(cfg.n_layers):
        x, _ = layer_forward(x, W[l + 1], cfg, cos, sin)
    y, _ = rmsnorm(x, W[-1]["final_norm"], cfg.rms_eps)
    z = y @ W[-1]["w_head"].T
    zmax = z.max(axis=1, keepdims=True)
    lse = zmax[:, 0] + np.log(np.sum(np.exp(z - zmax), axis=1))
    return float(np.mean(lse - z[np.arange(z.shape[0]), labels]))


def forward_backward(cfg: Config, weights, tokens, labels, dtype=np.float64, keep=False):
    """Loss and the gradient of every parameter for one batch.

    ``weights``: per block dicts of bfloat16 bit patterns (or float arrays).
    ``tokens``/``labels``: int arrays of B*s ids, token t = b*s + position.
    Returns (loss, grads) with grads shaped like ``weights`` in ``dtype``;
    with keep=True also a dict of intermediates (layer inputs, logits).
    """
    W = [{k: (bf16_bits_to_float(v, dtype) if v.dtype == np.uint16 else v.astype(dtype))
          for k, v in blk.items()} for blk in weights]
    L = cfg.n_layers
    tokens = np.asarray(tokens).reshape(-1)
    labels = np.asarray(labels).reshape(-1)
    cos, sin = rope_tables(cfg, dtype)
    x = W[0]["emb"][tokens]
    xs, caches = [], []
    for l in range(L):
        xs.append(x)
        x, c = layer_forward(x, W[l + 1], cfg, cos, sin)
        caches.append(c)
    loss, dx, ghead, z = head_forward_backward(x, W[L + 1], labels, cfg)
    grads = [None] * (L + 2)
    grads[L + 1] = ghead
    for l in reversed(range(L)):
        dx, grads[l + 1] = layer_backward(dx, caches[l], W[l + 1], cfg, cos, sin)
        caches[l] = None
    grads[0] = {"emb": embedding_backward(dx, tokens, cfg.vocab)}
    if keep:
        return loss, grads, {"x_in": xs, "x_final": x, "logits": z, "dx0": dx}
    return loss, grads


# ----------------------------------------------------------------------------
# Adam (reading R2), host-side as the chestersoft digest's Methodik places it
# ----------------------------------------------------------------------------
def adam_update(w_bits, g_bits, m, v, step, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, master=None):
    """One bias-corrected Adam step on stored values.

    w_bits, g_bits: bfloat16 bit patterns; m, v: float32. Arithmetic in float64;
    m and v are stored back as float32, w rounded to bfloat16 (nearest even).
    Returns (w_bits, m, v). With ``master`` (float32, R18) the step moves the
    master instead, which is stored as float32 and rounded to give w; returns
    (w_bits, m, v, master).
    """
    g = bf16_bits_to_float(g_bits)
    m64 = beta1 * m.astype(np.float64) + (1.0 - beta1) * g
    v64 = beta2 * v.astype(np.float64) + (1.0 - beta2) * g * g
    mhat = m64 / (1.0 - beta1 ** step)
    vhat = v64 / (1.0 - beta2 ** step)
    step_size = lr * mhat / (np.sqrt(vhat) + eps)
    if master is None:
        w_new = bf16_bits_to_float(w_bits) - step_size
        return float_to_bf16_bits(w_new), m64.astype(np.float32), v64.astype(np.float32)
    p_new = (master.astype(np.float64) - step_size).astype(np.float32)
    return float_to_bf16_bits(p_new.astype(np.float64)), m64.astype(np.float32), v64.astype(np.float32), p_new


def train_step(cfg: Config, arena: np.ndarray, tokens, labels, step: int, adam=None,
               dtype=np.float64, lay=None):
    """Plain definition of a training step on packed arena bytes (in place).

    Reads W, computes the loss and all gradients, writes G (bfloat16), then
    applies Adam to W, M, V with the stored G. Returns the loss.
    """
    lay = lay or layout(cfg)
    adam = adam or {}
    Wb = unpack_arena(cfg, arena, "W", lay)
    Gb = unpack_arena(cfg, arena, "G", lay)
    Mb = unpack_arena(cfg, arena, "M", lay)
    Vb = unpack_arena(cfg, arena, "V", lay)
    Pb = unpack_arena(cfg, arena, "P", lay) if cfg.fp32_master else None
    loss, grads = forward_backward(cfg, Wb, tokens, labels, dtype)
    for b in range(len(Wb)):
        for name in Wb[b]:
            Gb[b][name][...] = float_to_bf16_bits(grads[b][name])
            if Pb is None:
                w, m, v = adam_update(Wb[b][name], Gb[b][name], Mb[b][name], Vb[b][name], step, **adam)
            else:
                w, m, v, pm = adam_update(Wb[b][name], Gb[b][name], Mb[b][name], Vb[b][name], step, **adam,
                                          master=Pb[b][name])
                Pb[b][name][...] = pm
            Wb[b][name][...] = w
            Mb[b][name][...] = m
            Vb[b][name][...] = v
    return loss
