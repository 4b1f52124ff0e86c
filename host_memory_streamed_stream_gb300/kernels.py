"""Per-kernel binding (``include/mt_kernels.h``) over torch CUDA tensors: marshalling only.

Each function passes the tensors' device pointers and the current torch stream
to one C entry point and raises on a nonzero status.
"""
from __future__ import annotations

import torch

from . import MTError, _lib

EPI_STORE_BF16, EPI_STORE_F32, EPI_ADD_F32 = 0, 1, 2


def _p(t):
    return None if t is None else t.data_ptr()


def _s():
    return torch.cuda.current_stream().cuda_stream


def _ok(rc, what):
    if rc != 0:
        raise MTError(rc, what)


def gemm(A, a_mn, B, b_mn, M, N, K, epi=EPI_STORE_BF16, R=None, err=None, out=None):
    """C[M,N] = A * B (see mtk_gemm_bf16 for the operand storage orders)."""
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16 if epi == EPI_STORE_BF16 else torch.float32, device=A.device)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=A.device)
    _ok(_lib.load().mtk_gemm_bf16(A.data_ptr(), A.stride(0), int(a_mn), B.data_ptr(), B.stride(0), int(b_mn),
                                  out.data_ptr(), out.stride(0), _p(R), R.stride(0) if R is not None else 0, M, N, K,
                                  epi, err.data_ptr(), _s()), "gemm")
    return out


def gemm_use_workspace(device=None):
    """Give the mtk_gemm_* calls a zeroed split workspace on `device` (None: turn the split off).
    Returns the workspace tensor, which must stay alive while it is in use."""
    lib = _lib.load()
    if device is None:
        _ok(lib.mtk_gemm_use_workspace(None), "gemm_use_workspace")
        return None
    ws = torch.zeros(int(lib.mtk_gemm_workspace_bytes()), dtype=torch.uint8, device=device)
    _ok(lib.mtk_gemm_use_workspace(ws.data_ptr()), "gemm_use_workspace")
    return ws


def _err(err, dev):
    return torch.zeros(1, dtype=torch.int32, device=dev) if err is None else err


def gemm_qkv_rope(a, w, cos_sin, seq, n_heads, n_kv_heads, head_dim, err=None):
    """qkv = a W^T with RoPE on the q and k heads, fused in the GEMM epilogue."""
    T, h = a.shape
    qkv = torch.empty(T, (n_heads + 2 * n_kv_heads) * head_dim, dtype=torch.bfloat16, device=a.device)
    err = _err(err, a.device)
    _ok(_lib.load().mtk_gemm_qkv_rope(a.data_ptr(), w.data_ptr(), qkv.data_ptr(), cos_sin.data_ptr(), T, h, n_heads,
                                      n_kv_heads, head_dim, seq, err.data_ptr(), _s()), "gemm_qkv_rope")
    return qkv


def gemm_swiglu(b, wgu, f, keep_gu=False, err=None):
    """act = silu(b Wg^T) * (b Wu^T) fused in the GEMM epilogue; optionally also [g | u]."""
    T, h = b.shape
    act = torch.empty(T, f, dtype=torch.bfloat16, device=b.device)
    gu = torch.empty(T, 2 * f, dtype=torch.bfloat16, device=b.device) if keep_gu else None
    err = _err(err, b.device)
    _ok(_lib.load().mtk_gemm_swiglu(b.data_ptr(), wgu.data_ptr(), act.data_ptr(), _p(gu), T, h, f, err.data_ptr(),
                                    _s()), "gemm_swiglu")
    return act, gu


def gemm_swiglu_bwd(dy, wd, gu, f, err=None):
    """dgu from dact = dy Wd and gu = [g | u], the SwiGLU backward fused in the GEMM epilogue."""
    T, h = dy.shape
    dgu = torch.empty(T, 2 * f, dtype=torch.bfloat16, device=dy.device)
    err = _err(err, dy.device)
    _ok(_lib.load().mtk_gemm_swiglu_bwd(dy.data_ptr(), wd.data_ptr(), gu.data_ptr(), dgu.data_ptr(), T, h, f,
                                        err.data_ptr(), _s()), "gemm_swiglu_bwd")
    return dgu


def rmsnorm_fwd(x, gamma, eps=1e-5):
    T, h = x.shape
    y = torch.empty(T, h, dtype=torch.bfloat16, device=x.device)
    rstd = torch.empty(T, dtype=torch.float32, device=x.device)
    _ok(_lib.load().mtk_rmsnorm_fwd(x.data_ptr(), gamma.data_ptr(), y.data_ptr(), rstd.data_ptr(), T, h, eps, _s()),
        "rmsnorm_fwd")
    return y, rstd


def rmsnorm_bwd(dy, x, gamma, rstd, dres=None):
    T, h = x.shape
    lib = _lib.load()
    parts = lib.mtk_rmsnorm_bwd_parts(T)
    partial = torch.empty(parts, h, dtype=torch.float32, device=x.device)
    dx = torch.empty(T, h, dtype=torch.float32, device=x.device)
    dxb = torch.empty(T, h, dtype=torch.bfloat16, device=x.device)
    dg = torch.empty(h, dtype=torch.bfloat16, device=x.device)
    _ok(lib.mtk_rmsnorm_bwd(dy.data_ptr(), x.data_ptr(), gamma.data_ptr(), rstd.data_ptr(), _p(dres), dx.data_ptr(),
                            dxb.data_ptr(), partial.data_ptr(), dg.data_ptr(), T, h, _s()), "rmsnorm_bwd")
    return dx, dxb, dg


def rope_(qkv, seq, n_heads, n_kv_heads, head_dim, cos_sin, inverse=False):
    T = qkv.shape[0]
    _ok(_lib.load().mtk_rope(qkv.data_ptr(), qkv.stride(0), T, seq, n_heads, n_kv_heads, head_dim, cos_sin.data_ptr(),
                             int(inverse), _s()), "rope")
    return qkv


def swiglu_fwd(gu, f):
    T = gu.shape[0]
    act = torch.empty(T, f, dtype=torch.bfloat16, device=gu.device)
    _ok(_lib.load().mtk_swiglu_fwd(gu.data_ptr(), act.data_ptr(), T, f, _s()), "swiglu_fwd")
    return act


def swiglu_bwd(gu, dact, f):
    T = gu.shape[0]
    dgu = torch.empty(T, 2 * f, dtype=torch.bfloat16, device=gu.device)
    _ok(_lib.load().mtk_swiglu_bwd(gu.data_ptr(), dact.data_ptr(), dgu.data_ptr(), T, f, _s()), "swiglu_bwd")
    return dgu


def embed_fwd(tok, E):
    T = tok.numel()
    V, h = E.shape
    x = torch.empty(T, h, dtype=torch.float32, device=E.device)
    _ok(_lib.load().mtk_embed_fwd(tok.data_ptr(), E.data_ptr(), x.data_ptr(), T, h, _s()), "embed_fwd")
    return x


def embed_bwd(order, offsets, dx, V):
    h = dx.shape[1]
    dE = torch.empty(V, h, dtype=torch.bfloat16, device=dx.device)
    _ok(_lib.load().mtk_embed_bwd(order.data_ptr(), offsets.data_ptr(), dx.data_ptr(), dE.data_ptr(), V, h, _s()),
        "embed_bwd")
    return dE


def cross_entropy(logits, labels):
    T, V = logits.shape
    dl = torch.empty(T, V, dtype=torch.bfloat16, device=logits.device)
    rl = torch.empty(T, dtype=torch.float32, device=logits.device)
    loss = torch.empty(1, dtype=torch.float32, device=logits.device)
    _ok(_lib.load().mtk_cross_entropy(logits.data_ptr(), labels.data_ptr(), dl.data_ptr(), rl.data_ptr(),
                                      loss.data_ptr(), T, V, _s()), "cross_entropy")
    return loss, rl, dl


def attn_fwd(qkv, B, s, nh, nkv, hd, err=None):
    o = torch.empty(B * s, nh * hd, dtype=torch.bfloat16, device=qkv.device)
    lse = torch.empty(B, nh, s, dtype=torch.float32, device=qkv.device)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=qkv.device)
    _ok(_lib.load().mtk_attn_fwd(qkv.data_ptr(), o.data_ptr(), lse.data_ptr(), B, s, nh, nkv, hd, err.data_ptr(),
                                 _s()), "attn_fwd")
    return o, lse


def attn_bwd(qkv, o, lse, dout, B, s, nh, nkv, hd, err=None, cos_sin=None):
    """dqkv; with cos_sin (fp32 [s][hd/2][2]) dq and dk get the transpose RoPE rotation."""
    dqkv = torch.empty_like(qkv)
    delta = torch.empty(B, nh, (s + 127) // 128 * 128, 2, dtype=torch.float32, device=qkv.device)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=qkv.device)
    lib = _lib.load()
    if cos_sin is None:
        _ok(lib.mtk_attn_bwd(qkv.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(), dqkv.data_ptr(),
                             delta.data_ptr(), B, s, nh, nkv, hd, err.data_ptr(), _s()), "attn_bwd")
    else:
        _ok(lib.mtk_attn_bwd_rope(qkv.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(), dqkv.data_ptr(),
                                  delta.data_ptr(), cos_sin.data_ptr(), B, s, nh, nkv, hd, err.data_ptr(), _s()),
            "attn_bwd_rope")
    return dqkv
