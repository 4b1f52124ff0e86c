"""Cross-check the oracle against a model assembled from PyTorch CPU library routines.

torch.nn.functional's rms_norm, scaled_dot_product_attention (causal, GQA by
repeated heads), silu and cross_entropy, with gradients from autograd, all in
float64. This is an independent implementation of the same definition: a
transposed operand, a wrong scale or a wrong RoPE convention in the oracle
breaks the match.
"""
import numpy as np
import pytest

import oracle
import synth
from oracle import model as om

torch = pytest.importorskip("torch")
F = torch.nn.functional


def _torch_loss(cfg, Wt, tok, lab):
    B, s, h = cfg.batch, cfg.seq, cfg.hidden
    nh, nkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    inv = 1.0 / (cfg.rope_theta ** (torch.arange(0, hd, 2, dtype=torch.float64) / hd))
    ang = torch.outer(torch.arange(s, dtype=torch.float64), inv)
    cos = torch.cat([ang.cos(), ang.cos()], -1)
    sin = torch.cat([ang.sin(), ang.sin()], -1)

    def rot_half(x):
        x1, x2 = x[..., : hd // 2], x[..., hd // 2:]
        return torch.cat([-x2, x1], -1)

    x = Wt[0]["emb"][torch.as_tensor(tok, dtype=torch.long)].view(B, s, h)
    for l in range(cfg.n_layers):
        p = Wt[l + 1]
        a = F.rms_norm(x, (h,), p["attn_norm"], eps=cfg.rms_eps)
        q = (a @ p["wq"].T).view(B, s, nh, hd).transpose(1, 2)
        k = (a @ p["wk"].T).view(B, s, nkv, hd).transpose(1, 2)
        v = (a @ p["wv"].T).view(B, s, nkv, hd).transpose(1, 2)
        q = q * cos + rot_half(q) * sin
        k = k * cos + rot_half(k) * sin
        k = k.repeat_interleave(nh // nkv, dim=1)
        v = v.repeat_interleave(nh // nkv, dim=1)
        o = F.scaled_dot_product_attention(q, k, v, is_causal=True)
        x = x + o.transpose(1, 2).reshape(B, s, nh * hd) @ p["wo"].T
        b = F.rms_norm(x, (h,), p["ffn_norm"], eps=cfg.rms_eps)
        x = x + (F.silu(b @ p["wg"].T) * (b @ p["wu"].T)) @ p["wd"].T
    y = F.rms_norm(x, (h,), Wt[-1]["final_norm"], eps=cfg.rms_eps)
    z = (y @ Wt[-1]["w_head"].T).view(B * s, -1)
    return F.cross_entropy(z, torch.as_tensor(lab, dtype=torch.long))


@pytest.mark.parametrize("cfg", [
    oracle.Config(n_layers=2, hidden=256, n_heads=4, n_kv_heads=4, ffn=1024, vocab=1024, seq=128, batch=2),
    oracle.Config(n_layers=2, hidden=128, n_heads=4, n_kv_heads=2, ffn=344, vocab=500, seq=48, batch=3),
], ids=["tiny", "gqa_ragged"])
def test_oracle_matches_torch_autograd(cfg):
    Wb = oracle.init_params(cfg, synth, synth.WEIGHT_SEED)
    tok = synth.tokens(cfg.tokens, cfg.vocab)
    lab = synth.labels(cfg.tokens, cfg.vocab)
    loss, grads = oracle.forward_backward(cfg, Wb, tok, lab, np.float64)
    Wt = [{k: torch.tensor(om.bf16_bits_to_float(v), requires_grad=True) for k, v in blk.items()} for blk in Wb]
    lt = _torch_loss(cfg, Wt, tok, lab)
    lt.backward()
    assert abs(lt.item() - loss) < 1e-12 * abs(loss)
    for b in range(cfg.n_layers + 2):
        for k, t in Wt[b].items():
            ref = t.grad.numpy()
            err = np.max(np.abs(grads[b][k] - ref)) / np.max(np.abs(ref))
            assert err < 1e-10, (b, k, err)
