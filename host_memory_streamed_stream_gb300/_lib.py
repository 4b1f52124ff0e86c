"""ctypes loader of ``libmt.so`` with the signatures of ``include/mt.h`` and ``include/mt_kernels.h``.

The library is built in-tree (``_build.build()``). There is no fallback: if the
shared library is missing or does not load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmt.so")

c_int, c_i32, c_i64, c_u32, c_u64, c_f32, c_vp = (ctypes.c_int, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32,
                                                  ctypes.c_uint64, ctypes.c_float, ctypes.c_void_p)
P = ctypes.POINTER


class ModelCfg(ctypes.Structure):
    _fields_ = [("n_layers", c_i32), ("hidden", c_i32), ("n_heads", c_i32), ("n_kv_heads", c_i32), ("ffn", c_i32),
                ("vocab", c_i32), ("seq", c_i32), ("batch", c_i32), ("rms_eps", c_f32), ("rope_theta", c_f32),
                ("flags", c_u32)]


class DeviceResources(ctypes.Structure):
    _fields_ = [("workspace", c_vp), ("workspace_bytes", c_u64), ("streams", c_vp * 3)]


class AdamCfg(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("step", c_i64)]


class Stats(ctypes.Structure):
    _fields_ = [("step_ms", ctypes.c_double), ("compute_busy_ms", ctypes.c_double),
                ("h2d_busy_ms", ctypes.c_double), ("d2h_busy_ms", ctypes.c_double),
                ("exposed_ms", ctypes.c_double), ("fwd_ms", ctypes.c_double), ("bwd_ms", ctypes.c_double),
                ("adam_ms", ctypes.c_double), ("host_step_ms", ctypes.c_double), ("h2d_bytes", c_u64),
                ("d2h_bytes", c_u64), ("kernel_launches", c_i64), ("steps", c_i64),
                ("copy_bytes", (c_u64 * 2) * 2), ("copy_ms", (ctypes.c_double * 2) * 2),
                ("first_copy_ms", ctypes.c_double), ("embed_gather_gbs", ctypes.c_double),
                ("sparse_embed", c_i32)]


class BlockLayout(ctypes.Structure):
    _fields_ = [("offset", c_u64), ("bytes", c_u64), ("n_tensors", c_i32), ("n_sections", c_i32),
                ("section_offset", c_u64 * 5), ("section_bytes", c_u64 * 5), ("tensor_offset", (c_u64 * 9) * 5),
                ("rows", c_i64 * 9), ("cols", c_i64 * 9)]


class Layout(ctypes.Structure):
    _fields_ = [("total_bytes", c_u64), ("max_w_section", c_u64), ("n_blocks", c_i32), ("n_sections", c_i32),
                ("capacity", c_i32), ("blocks", P(BlockLayout))]


class HostAllocInfo(ctypes.Structure):
    _fields_ = [("chunk_bytes", c_u64), ("chunks", c_i32), ("spare", c_i32), ("slow_found", c_i32),
                ("replaced", c_i32), ("median_gbs", ctypes.c_double), ("min_gbs", ctypes.c_double)]


class KernelStats(ctypes.Structure):
    _fields_ = [("launches", c_i64), ("ms", ctypes.c_double), ("flops", ctypes.c_double),
                ("bytes", ctypes.c_double)]


# name -> (restype, argtypes)
SIGNATURES = {
    # mt.h
    "mt_arena_layout": (c_int, [P(ModelCfg), P(Layout)]),
    "mt_arena_bytes": (c_int, [P(ModelCfg), P(c_u64)]),
    "mt_block_count": (c_int, [P(ModelCfg), P(c_i32)]),
    "mt_tensor_count": (c_int, [P(ModelCfg), c_i32, P(c_i32)]),
    "mt_block_offset": (c_int, [P(ModelCfg), c_i32, P(c_u64), P(c_u64)]),
    "mt_tensor_offset": (c_int, [P(ModelCfg), c_i32, c_i32, c_i32, P(c_u64), P(c_i64), P(c_i64), P(c_i32)]),
    "mt_host_alloc": (c_int, [c_u64, P(c_vp)]),
    "mt_host_free": (c_int, [c_vp]),
    "mt_host_alloc_query": (c_int, [c_vp, P(HostAllocInfo)]),
    "mt_workspace_bytes": (c_int, [P(ModelCfg), P(c_u64)]),
    "mt_create": (c_int, [P(ModelCfg), P(DeviceResources), P(c_vp)]),
    "mt_bind_host_arena": (c_int, [c_vp, c_vp, c_u64]),
    "mt_train_step": (c_int, [c_vp, c_vp, c_vp, P(c_f32)]),
    "mt_adam_step": (c_int, [c_vp, P(AdamCfg)]),
    "mt_train_step_adam": (c_int, [c_vp, c_vp, c_vp, P(AdamCfg), P(c_f32)]),
    "mt_adam_apply": (c_int, [P(ModelCfg), c_vp, c_u64, P(AdamCfg)]),
    "mt_host_bandwidth": (c_int, [c_u64, c_i32, P(ctypes.c_double), P(c_i32)]),
    "mt_get_stats": (c_int, [c_vp, P(Stats)]),
    "mt_get_kernel_stats": (c_int, [c_vp, c_i32, P(KernelStats)]),
    "mt_set_kernel_timing": (c_int, [c_vp, c_i32]),
    "mt_read_checkpoint": (c_int, [c_vp, c_i32, c_vp]),
    "mt_capture_input_grad": (c_int, [c_vp, c_i32, c_vp]),
    "mt_set_head_chunk_rows": (c_int, [c_vp, c_i32]),
    "mt_master_init": (c_int, [P(ModelCfg), c_vp, c_u64]),
    "mt_last_error": (ctypes.c_char_p, [c_vp]),
    "mt_destroy": (None, [c_vp]),
    # mt_kernels.h
    "mtk_gemm_bf16": (c_int, [c_vp, c_i64, c_int, c_vp, c_i64, c_int, c_vp, c_i64, c_vp, c_i64, c_int, c_int, c_int,
                              c_int, c_vp, c_vp]),
    "mtk_gemm_workspace_bytes": (c_u64, []),
    "mtk_gemm_workspace_clear_bytes": (c_u64, []),
    "mtk_gemm_use_workspace": (c_int, [c_vp]),
    "mtk_gemm_qkv_rope": (c_int, [c_vp, c_vp, c_vp, c_vp, c_int, c_int, c_int, c_int, c_int, c_int, c_vp, c_vp]),
    "mtk_gemm_swiglu": (c_int, [c_vp, c_vp, c_vp, c_vp, c_int, c_int, c_int, c_vp, c_vp]),
    "mtk_gemm_swiglu_bwd": (c_int, [c_vp, c_vp, c_vp, c_vp, c_int, c_int, c_int, c_vp, c_vp]),
    "mtk_rmsnorm_fwd": (c_int, [c_vp, c_vp, c_vp, c_vp, c_int, c_int, c_f32, c_vp]),
    "mtk_rmsnorm_bwd_parts": (c_int, [c_int]),
    "mtk_rmsnorm_bwd": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_int, c_int, c_vp]),
    "mtk_rmsnorm_bwd_noalloc": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_int, c_int, c_vp]),
    "mtk_rope": (c_int, [c_vp, c_i64, c_int, c_int, c_int, c_int, c_int, c_vp, c_int, c_vp]),
    "mtk_swiglu_fwd": (c_int, [c_vp, c_vp, c_int, c_int, c_vp]),
    "mtk_swiglu_bwd": (c_int, [c_vp, c_vp, c_vp, c_int, c_int, c_vp]),
    "mtk_embed_fwd": (c_int, [c_vp, c_vp, c_vp, c_int, c_int, c_vp]),
    "mtk_embed_bwd": (c_int, [c_vp, c_vp, c_vp, c_vp, c_int, c_int, c_vp]),
    "mtk_cross_entropy": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_int, c_int, c_vp]),
    "mtk_attn_fwd": (c_int, [c_vp, c_vp, c_vp, c_int, c_int, c_int, c_int, c_int, c_vp, c_vp]),
    "mtk_attn_bwd": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_int, c_int, c_int, c_int, c_int, c_vp, c_vp]),
    "mtk_attn_bwd_rope": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_int, c_int, c_int, c_int, c_int, c_vp,
                                  c_vp]),
    "mtk_attn_block_slot": (c_int, [c_int, c_int, c_int, P(c_int), P(c_int)]),
    "mtk_bounded_wait_check": (c_int, [c_vp, c_vp, c_i64, c_vp]),
}

_lib = None


def load() -> ctypes.CDLL:
    """Load ``libmt.so`` (raises OSError if it has not been built or cannot load)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise OSError(f"{LIB_PATH} is missing: build it with host_memory_streamed_stream_gb300._build.build()")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
    return _lib
