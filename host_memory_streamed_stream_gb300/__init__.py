"""Layer-streamed full-precision training step on one GB300 (Python binding).

A thin binding over ``libmt.so`` (C ABI in ``include/mt.h``): argument
marshalling only. Every step of the training path runs in the library's CUDA
kernels and its C++ host runtime; PyTorch supplies device memory and streams.
There is no CPU or eager fallback: if the library is missing, importing a
function that needs it raises.

Method: "MegaTrain: Full Precision Training of 100B+ Parameter Large Language
Models on a Single GPU" — parameters, gradients and Adam states in a pinned
host arena of 4 KB-aligned per-layer blocks; the GPU receives one layer's
weights at a time over three CUDA streams with double buffering (chatpaper
abstract; chestersoft digest, Methodik).
"""
from __future__ import annotations

import ctypes
import dataclasses

import numpy as np

from . import _lib

SEC_W, SEC_G, SEC_M, SEC_V, SEC_P = 0, 1, 2, 3, 4
FLAG_RESIDENT, FLAG_OFFLOAD_CKPT, FLAG_SINGLE_BUFFER, FLAG_KERNEL_TIMING, FLAG_FP32_MASTER = 1, 2, 4, 8, 16
FLAG_DENSE_EMBED = 32
KIND_NAMES = ["gemm", "attn_fwd", "attn_bwd", "pointwise", "cross_entropy", "embed"]
ERRORS = {-1: "MT_EINVAL", -2: "MT_ENOMEM", -3: "MT_EALIGN", -4: "MT_ESTATE", -5: "MT_ECUDA", -6: "MT_ETIMEOUT",
          -7: "MT_EKERNEL"}


class MTError(RuntimeError):
    def __init__(self, code: int, msg: str = ""):
        self.code = code
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")


def _check(code: int, ctx=None):
    if code != 0:
        msg = _lib.load().mt_last_error(ctx)
        raise MTError(code, msg.decode() if msg else "")


@dataclasses.dataclass(frozen=True)
class ModelConfig:
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
    flags: int = 0

    @property
    def head_dim(self) -> int:
        return self.hidden // self.n_heads

    @property
    def tokens(self) -> int:
        return self.batch * self.seq

    def c(self) -> _lib.ModelCfg:
        return _lib.ModelCfg(self.n_layers, self.hidden, self.n_heads, self.n_kv_heads, self.ffn, self.vocab,
                             self.seq, self.batch, self.rms_eps, self.rope_theta, self.flags)

    def with_flags(self, flags: int) -> "ModelConfig":
        return dataclasses.replace(self, flags=flags)

    def params(self) -> int:
        h, f, V, L = self.hidden, self.ffn, self.vocab, self.n_layers
        qd, kvd = self.n_heads * self.head_dim, self.n_kv_heads * self.head_dim
        return 2 * V * h + h + L * (2 * h + qd * h + 2 * kvd * h + h * qd + 3 * f * h)


# ---------------------------------------------------------------------------- layout
def arena_bytes(cfg: ModelConfig) -> int:
    out = ctypes.c_uint64()
    _check(_lib.load().mt_arena_bytes(ctypes.byref(cfg.c()), ctypes.byref(out)))
    return out.value


def arena_layout(cfg: ModelConfig) -> dict:
    """The whole packed-block layout from one mt_arena_layout call (two: counts, then blocks).
    Returns {"total", "max_w_section", "n_sections", "blocks": [{"offset", "bytes", "sections":
    [(offset, bytes)], "tensors": [[offset per tensor] per section], "shapes": [(rows, cols)]}]}."""
    lib = _lib.load()
    lay = _lib.Layout()
    lay.capacity = 0
    _check(lib.mt_arena_layout(ctypes.byref(cfg.c()), ctypes.byref(lay)))
    arr = (_lib.BlockLayout * lay.n_blocks)()
    lay.capacity = lay.n_blocks
    lay.blocks = arr
    _check(lib.mt_arena_layout(ctypes.byref(cfg.c()), ctypes.byref(lay)))
    blocks = []
    for b in arr:
        ns, nt = b.n_sections, b.n_tensors
        blocks.append({"offset": b.offset, "bytes": b.bytes,
                       "sections": [(b.section_offset[s], b.section_bytes[s]) for s in range(ns)],
                       "tensors": [[b.tensor_offset[s][t] for t in range(nt)] for s in range(ns)],
                       "shapes": [(b.rows[t], b.cols[t]) for t in range(nt)]})
    return {"total": lay.total_bytes, "max_w_section": lay.max_w_section, "n_sections": lay.n_sections,
            "blocks": blocks}


def workspace_bytes(cfg: ModelConfig) -> int:
    out = ctypes.c_uint64()
    _check(_lib.load().mt_workspace_bytes(ctypes.byref(cfg.c()), ctypes.byref(out)))
    return out.value


def num_blocks(cfg: ModelConfig) -> int:
    return cfg.n_layers + 2


def num_tensors(cfg: ModelConfig, block: int) -> int:
    out = ctypes.c_int32()
    _check(_lib.load().mt_tensor_count(ctypes.byref(cfg.c()), block, ctypes.byref(out)))
    return out.value


def tensor_offset(cfg: ModelConfig, block: int, section: int, tensor: int):
    """(byte offset from the arena base, rows, cols, element bytes)."""
    off, rows, cols, esz = ctypes.c_uint64(), ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32()
    _check(_lib.load().mt_tensor_offset(ctypes.byref(cfg.c()), block, section, tensor, ctypes.byref(off),
                                        ctypes.byref(rows), ctypes.byref(cols), ctypes.byref(esz)))
    return off.value, rows.value, cols.value, esz.value


def block_offset(cfg: ModelConfig, block: int):
    off, nb = ctypes.c_uint64(), ctypes.c_uint64()
    _check(_lib.load().mt_block_offset(ctypes.byref(cfg.c()), block, ctypes.byref(off), ctypes.byref(nb)))
    return off.value, nb.value


def weight_tensors(cfg: ModelConfig):
    """(block, tensor index, W-section byte offset, numel, is_gain) for every tensor."""
    out = []
    for b in range(num_blocks(cfg)):
        for t in range(num_tensors(cfg, b)):
            off, rows, cols, _ = tensor_offset(cfg, b, SEC_W, t)
            out.append((b, t, off, rows * cols, cols == 1))
    return out


# ---------------------------------------------------------------------------- host arena
class HostArena:
    """Page-locked host memory holding the packed blocks (owned by this object)."""

    def __init__(self, nbytes: int, pinned: bool = True):
        self.nbytes = int(nbytes)
        self._pinned = pinned
        if pinned:
            p = ctypes.c_void_p()
            _check(_lib.load().mt_host_alloc(self.nbytes, ctypes.byref(p)))
            self.ptr = p.value
            self._keep = None
        else:  # plain 4096-aligned host memory (the library registers it on bind)
            raw = np.empty(self.nbytes + 4096, dtype=np.uint8)
            start = (-raw.ctypes.data) % 4096
            self._keep = raw
            self.ptr = raw.ctypes.data + start
        self.array = np.ctypeslib.as_array((ctypes.c_uint8 * self.nbytes).from_address(self.ptr))

    def info(self) -> dict | None:
        """What the allocator found for huge-page backed memory (None otherwise): huge pages,
        spares, pages found slow and swapped, and the per-page host-to-device GB/s."""
        if not (self.ptr and self._pinned):
            return None
        i = _lib.HostAllocInfo()
        if _lib.load().mt_host_alloc_query(self.ptr, ctypes.byref(i)) != 0:
            return None
        return {"huge_page_bytes": i.chunk_bytes, "huge_pages": i.chunks, "spare": i.spare,
                "slow_found": i.slow_found, "replaced": i.replaced, "median_gbs": round(i.median_gbs, 1),
                "min_gbs": round(i.min_gbs, 1)}

    def free(self):
        if self.ptr and self._pinned:
            _lib.load().mt_host_free(self.ptr)
        self.ptr = 0
        self.array = None
        self._keep = None


def master_init(cfg: ModelConfig, arena: HostArena):
    """With FLAG_FP32_MASTER: set the fp32 master section P to the bf16 weights W."""
    _check(_lib.load().mt_master_init(ctypes.byref(cfg.c()), arena.ptr, arena.nbytes))


def adam_apply(cfg: ModelConfig, arena: HostArena, step: int, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8):
    """Host Adam on an arena without a GPU context."""
    hp = _lib.AdamCfg(lr, beta1, beta2, eps, step)
    _check(_lib.load().mt_adam_apply(ctypes.byref(cfg.c()), arena.ptr, arena.nbytes, ctypes.byref(hp)))


def host_bandwidth(nbytes: int = 3 << 30, reps: int = 5):
    """(GB/s, threads) of a host triad over nbytes in all (the host Adam's memory roofline)."""
    gbs, th = ctypes.c_double(), ctypes.c_int32()
    _check(_lib.load().mt_host_bandwidth(int(nbytes), int(reps), ctypes.byref(gbs), ctypes.byref(th)))
    return gbs.value, th.value


# ---------------------------------------------------------------------------- training context
class Trainer:
    """One mt_ctx: device buffers and streams from PyTorch, the arena from the caller (or allocated)."""

    def __init__(self, cfg: ModelConfig, arena: HostArena | None = None, torch_resources: bool = True):
        import torch  # device memory and streams only

        self.cfg = cfg
        self.lib = _lib.load()
        self._torch = torch
        res = None
        self._ws = None
        self._streams = []
        if torch_resources:
            nbytes = workspace_bytes(cfg)
            self._ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
            self._streams = [torch.cuda.Stream() for _ in range(3)]
            res = _lib.DeviceResources(self._ws.data_ptr(), nbytes,
                                       (ctypes.c_void_p * 3)(*[s.cuda_stream for s in self._streams]))
        ctx = ctypes.c_void_p()
        _check(self.lib.mt_create(ctypes.byref(cfg.c()), ctypes.byref(res) if res else None, ctypes.byref(ctx)))
        self.ctx = ctx
        self._own_arena = arena is None
        self.arena = arena if arena is not None else HostArena(arena_bytes(cfg))
        _check(self.lib.mt_bind_host_arena(self.ctx, self.arena.ptr, self.arena.nbytes), self.ctx)
        self._loss = ctypes.c_float()

    def step(self, tokens: np.ndarray, labels: np.ndarray) -> float:
        tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(-1)
        labels = np.ascontiguousarray(labels, dtype=np.int32).reshape(-1)
        if tokens.size != self.cfg.tokens or labels.size != self.cfg.tokens:
            raise MTError(-1, "tokens/labels must hold batch*seq ids")
        _check(self.lib.mt_train_step(self.ctx, tokens.ctypes.data, labels.ctypes.data, ctypes.byref(self._loss)),
               self.ctx)
        return float(self._loss.value)

    def step_adam(self, tokens: np.ndarray, labels: np.ndarray, step: int, lr=1e-3, beta1=0.9, beta2=0.999,
                  eps=1e-8) -> float:
        """Training step with the host Adam update overlapped with the backward pass."""
        tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(-1)
        labels = np.ascontiguousarray(labels, dtype=np.int32).reshape(-1)
        if tokens.size != self.cfg.tokens or labels.size != self.cfg.tokens:
            raise MTError(-1, "tokens/labels must hold batch*seq ids")
        hp = _lib.AdamCfg(lr, beta1, beta2, eps, step)
        _check(self.lib.mt_train_step_adam(self.ctx, tokens.ctypes.data, labels.ctypes.data, ctypes.byref(hp),
                                           ctypes.byref(self._loss)), self.ctx)
        return float(self._loss.value)

    def adam(self, step: int, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8):
        hp = _lib.AdamCfg(lr, beta1, beta2, eps, step)
        _check(self.lib.mt_adam_step(self.ctx, ctypes.byref(hp)), self.ctx)

    def stats(self) -> dict:
        s = _lib.Stats()
        _check(self.lib.mt_get_stats(self.ctx, ctypes.byref(s)), self.ctx)
        out = {}
        for k, _ in _lib.Stats._fields_:
            v = getattr(s, k)
            out[k] = [[v[i][j] for j in range(2)] for i in range(2)] if k in ("copy_bytes", "copy_ms") else v
        return out

    def read_checkpoint(self, layer: int) -> np.ndarray:
        """Layer-boundary activation x_layer (fp32 [batch*seq, hidden]) of the last step."""
        out = np.empty((self.cfg.tokens, self.cfg.hidden), dtype=np.float32)
        _check(self.lib.mt_read_checkpoint(self.ctx, layer, out.ctypes.data), self.ctx)
        return out

    def capture_input_grad(self, layer: int) -> np.ndarray:
        """Arm a copy of dL/dx_layer (fp32 [batch*seq, hidden]) during later steps; returns the
        array (page-locked) that holds it after each step."""
        nbytes = self.cfg.tokens * self.cfg.hidden * 4
        buf = HostArena(nbytes)
        self._captures = getattr(self, "_captures", {})
        old = self._captures.get(layer)
        _check(self.lib.mt_capture_input_grad(self.ctx, layer, buf.ptr), self.ctx)
        self._captures[layer] = buf
        if old is not None:
            old.free()
        return buf.array.view(np.float32).reshape(self.cfg.tokens, self.cfg.hidden)

    def clear_captures(self):
        _check(self.lib.mt_capture_input_grad(self.ctx, -1, None), self.ctx)
        for b in getattr(self, "_captures", {}).values():
            b.free()
        self._captures = {}

    def set_head_chunk_rows(self, rows: int):
        """Token rows per LM-head chunk for later steps (0: the default)."""
        _check(self.lib.mt_set_head_chunk_rows(self.ctx, int(rows)), self.ctx)

    def set_kernel_timing(self, on: bool):
        _check(self.lib.mt_set_kernel_timing(self.ctx, 1 if on else 0), self.ctx)

    def kernel_stats(self) -> dict:
        out = {}
        for i, name in enumerate(KIND_NAMES):
            k = _lib.KernelStats()
            _check(self.lib.mt_get_kernel_stats(self.ctx, i, ctypes.byref(k)), self.ctx)
            out[name] = {"launches": k.launches, "ms": k.ms, "flops": k.flops, "bytes": k.bytes}
        return out

    def compute_stream(self):
        return self._streams[1] if self._streams else None

    def close(self):
        if getattr(self, "ctx", None):
            self.lib.mt_destroy(self.ctx)
            self.ctx = None
        for b in getattr(self, "_captures", {}).values():
            b.free()
        self._captures = {}
        if self._own_arena and self.arena is not None:
            self.arena.free()
            self.arena = None
        self._ws = None

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def fill_synthetic(cfg: ModelConfig, arena: HostArena, gen, seed: int, std: float = 0.02):
    """Write the initial state into an arena with the seeded generator module ``gen``
    (``synth``): gains 1.0, matrices N(0, std^2) bf16; G, M, V zero; with FLAG_FP32_MASTER the
    master section P equal to W."""
    gen.zero_into(arena.ptr, arena.nbytes)
    for b, t, off, n, is_gain in weight_tensors(cfg):
        if is_gain:
            gen.const_bf16_into(arena.ptr + off, n, 1.0)
        else:
            gen.normal_bf16_into(arena.ptr + off, n, seed, gen.weight_stream(b, t), std)
    if cfg.flags & FLAG_FP32_MASTER:
        master_init(cfg, arena)


def section_view(cfg: ModelConfig, arena: HostArena, block: int, section: int, tensor: int) -> np.ndarray:
    """numpy view of one tensor of the arena (uint16 bf16 bits for W/G, float32 for M/V/P)."""
    off, rows, cols, esz = tensor_offset(cfg, block, section, tensor)
    dt = np.uint16 if esz == 2 else np.float32
    v = arena.array[off:off + rows * cols * esz].view(dt)
    return v.reshape(rows) if cols == 1 else v.reshape(rows, cols)
