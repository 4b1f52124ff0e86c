"""CPU checks of the C ABI: the library loads, exports every declared symbol, its
layout equals the oracle's independent layout, its packing is bit-exact, its host
Adam matches the oracle's, and its argument checks reject bad input."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def mt():
    from host_memory_streamed_stream_gb300 import _build

    _build.build()
    import host_memory_streamed_stream_gb300 as m

    m._lib.load()
    return m


CFGS = {
    "tiny": dict(n_layers=2, hidden=256, n_heads=4, n_kv_heads=4, ffn=1024, vocab=1024, seq=128, batch=2),
    "gqa_ragged": dict(n_layers=3, hidden=512, n_heads=4, n_kv_heads=2, ffn=1368, vocab=1000, seq=200, batch=2),
    "1.3b": dict(n_layers=24, hidden=2048, n_heads=16, n_kv_heads=16, ffn=5504, vocab=32000, seq=2048, batch=4),
    "7b": dict(n_layers=32, hidden=4096, n_heads=32, n_kv_heads=32, ffn=11008, vocab=32000, seq=4096, batch=2),
    "14b": dict(n_layers=48, hidden=5120, n_heads=40, n_kv_heads=8, ffn=13824, vocab=152064, seq=4096, batch=1),
    "7b_long": dict(n_layers=32, hidden=4096, n_heads=32, n_kv_heads=32, ffn=11008, vocab=32000, seq=131072,
                    batch=1),
}


def _declared_functions():
    names = set()
    for hdr in ("mt.h", "mt_kernels.h"):
        text = open(os.path.join(ROOT, "include", hdr)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*(mtk?_[a-z0-9_]+)\s*\(", text, re.M):
            names.add(m.group(1))
    return names


def test_library_exports_every_declared_symbol(mt):
    lib = ctypes.CDLL(mt._lib.LIB_PATH)
    names = _declared_functions()
    assert len(names) >= 25
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding declares a signature for each of them
    assert names == set(mt._lib.SIGNATURES)


@pytest.mark.parametrize("name", list(CFGS))
def test_layout_matches_oracle(mt, name):
    cfg = mt.ModelConfig(**CFGS[name])
    ocfg = oracle.Config(**CFGS[name])
    lay = oracle.layout(ocfg)
    assert mt.arena_bytes(cfg) == lay["total"]
    for b, blk in enumerate(lay["blocks"]):
        assert mt.block_offset(cfg, b) == (blk["offset"], blk["bytes"])
        tensors = oracle.model.block_tensors(ocfg, b)
        assert mt.num_tensors(cfg, b) == len(tensors)
        for si, sec in enumerate("WGMV"):
            for ti, (tname, shape) in enumerate(tensors):
                off, rows, cols, esz = mt.tensor_offset(cfg, b, si, ti)
                assert off == blk["sections"][sec]["tensors"][tname], (b, sec, tname)
                assert (rows, cols) == (shape[0], shape[1] if len(shape) == 2 else 1)
                assert esz == (2 if sec in "WG" else 4)


@pytest.mark.parametrize("name", ["tiny", "gqa_ragged", "14b"])
def test_arena_layout_call_matches_oracle(mt, name):
    """mt_arena_layout (the whole layout in one call) equals the oracle's independent layout."""
    cfg, ocfg = mt.ModelConfig(**CFGS[name]), oracle.Config(**CFGS[name])
    lay, got = oracle.layout(ocfg), mt.arena_layout(cfg)
    assert got["total"] == lay["total"]
    assert got["n_sections"] == 4 and len(got["blocks"]) == cfg.n_layers + 2
    assert got["max_w_section"] == max(blk["sections"]["W"]["bytes"] for blk in lay["blocks"])
    for b, (blk, g) in enumerate(zip(lay["blocks"], got["blocks"])):
        assert (g["offset"], g["bytes"]) == (blk["offset"], blk["bytes"])
        tensors = oracle.model.block_tensors(ocfg, b)
        assert g["shapes"] == [(sh[0], sh[1] if len(sh) == 2 else 1) for _, sh in tensors]
        for si, sec in enumerate("WGMV"):
            assert g["sections"][si] == (blk["sections"][sec]["offset"], blk["sections"][sec]["bytes"])
            assert g["tensors"][si] == [blk["sections"][sec]["tensors"][t] for t, _ in tensors]


def test_arena_layout_partial_capacity_and_errors(mt):
    import ctypes as C

    lib = mt._lib.load()
    cfg = mt.ModelConfig(**CFGS["tiny"])
    lay = mt._lib.Layout()
    lay.capacity = 1
    one = (mt._lib.BlockLayout * 1)()
    lay.blocks = one
    assert lib.mt_arena_layout(C.byref(cfg.c()), C.byref(lay)) == 0
    assert lay.n_blocks == 4 and one[0].n_tensors == 1 and one[0].offset == 0
    lay.capacity = -1
    assert lib.mt_arena_layout(C.byref(cfg.c()), C.byref(lay)) == -1
    lay.capacity, lay.blocks = 2, None
    assert lib.mt_arena_layout(C.byref(cfg.c()), C.byref(lay)) == -1
    bad = mt.ModelConfig(**dict(CFGS["tiny"], hidden=100))
    lay.capacity = 0
    assert lib.mt_arena_layout(C.byref(bad.c()), C.byref(lay)) == -1
    assert lib.mt_arena_layout(C.byref(cfg.c()), None) == -1


def test_packing_bit_exact(mt):
    """The product's arena fill (its layout + the shared generator) equals the oracle's re-pack."""
    kw = CFGS["gqa_ragged"]
    cfg, ocfg = mt.ModelConfig(**kw), oracle.Config(**kw)
    arena = mt.HostArena(mt.arena_bytes(cfg), pinned=False)
    arena.array[:] = 0xAB  # garbage first: the fill must write every byte that matters
    mt.fill_synthetic(cfg, arena, synth, synth.WEIGHT_SEED)
    ref = oracle.pack_arena(ocfg, oracle.init_params(ocfg, synth, synth.WEIGHT_SEED))
    assert arena.array.tobytes() == ref.tobytes()


def _random_arena(mt, cfg, ocfg, seed):
    arena = mt.HostArena(mt.arena_bytes(cfg), pinned=False)
    mt.fill_synthetic(cfg, arena, synth, synth.WEIGHT_SEED)
    rng = np.random.default_rng(seed)
    for blk in oracle.unpack_arena(ocfg, arena.array, "G"):
        for v in blk.values():
            v[...] = oracle.float_to_bf16_bits(rng.standard_normal(v.shape) * 1e-3)
    for sec, scale in (("M", 1e-3), ("V", 1e-6)):
        for blk in oracle.unpack_arena(ocfg, arena.array, sec):
            for v in blk.values():
                v[...] = (np.abs(rng.standard_normal(v.shape)) * scale).astype(np.float32)
    return arena


@pytest.mark.parametrize("step", [1, 2, 7])
def test_host_adam_matches_oracle(mt, step):
    kw = CFGS["tiny"]
    cfg, ocfg = mt.ModelConfig(**kw), oracle.Config(**kw)
    arena = _random_arena(mt, cfg, ocfg, seed=step)
    before = arena.array.copy()
    mt.adam_apply(cfg, arena, step)
    W0, G0, M0, V0 = (oracle.unpack_arena(ocfg, before, s) for s in "WGMV")
    W1, M1, V1 = (oracle.unpack_arena(ocfg, arena.array, s) for s in "WMV")
    for b in range(len(W0)):
        for k in W0[b]:
            w, m, v = oracle.adam_update(W0[b][k], G0[b][k], M0[b][k], V0[b][k], step)
            # fp32 arithmetic: error a few ulp of the operands (m0, g ~ 1e-3; v0, g^2 ~ 1e-6), and
            # the sums may cancel, so the bound is absolute at the operands' scale
            m_scale = 0.9 * np.abs(M0[b][k]) + 0.1 * np.abs(oracle.bf16_bits_to_float(G0[b][k]))
            v_scale = 0.999 * np.abs(V0[b][k]) + 0.001 * oracle.bf16_bits_to_float(G0[b][k]) ** 2
            assert np.all(np.abs(M1[b][k] - m) <= 4.8e-7 * m_scale + 1e-30), (b, k)
            assert np.all(np.abs(V1[b][k] - v) <= 4.8e-7 * v_scale + 1e-30), (b, k)
            # fp32 vs float64 arithmetic may land on the other side of a bf16 rounding boundary:
            # at most one bf16 step of the result, plus 1e-4 lr for the fp32 error of the update
            # itself (m may have cancelled, see above) when w' is near zero
            got = oracle.bf16_bits_to_float(W1[b][k])
            ref = oracle.bf16_bits_to_float(w)
            assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-7), (b, k)
            assert np.mean(W1[b][k] != w) < 1e-2


def test_host_adam_closed_form(mt):
    """Product Adam on hand-set values: w = 0.5, g = bf16(0.1), t = 1 -> bf16 0.498046875."""
    kw = CFGS["tiny"]
    cfg, ocfg = mt.ModelConfig(**kw), oracle.Config(**kw)
    arena = mt.HostArena(mt.arena_bytes(cfg), pinned=False)
    arena.array[:] = 0
    W = oracle.unpack_arena(ocfg, arena.array, "W")
    G = oracle.unpack_arena(ocfg, arena.array, "G")
    W[1]["wq"][0, 0] = oracle.float_to_bf16_bits(np.array(0.5))
    G[1]["wq"][0, 0] = oracle.float_to_bf16_bits(np.array(0.1))
    W[1]["wq"][0, 1] = oracle.float_to_bf16_bits(np.array(-0.02))
    G[1]["wq"][0, 1] = oracle.float_to_bf16_bits(np.array(-3e-4))
    W[1]["wq"][0, 2] = oracle.float_to_bf16_bits(np.array(0.375))
    mt.adam_apply(cfg, arena, 1)
    vals = oracle.bf16_bits_to_float(W[1]["wq"][0, :3])
    assert list(vals) == [0.498046875, -0.01904296875, 0.375]


def test_config_validation(mt):
    bad = dict(CFGS["tiny"], hidden=200)
    with pytest.raises(mt.MTError) as e:
        mt.arena_bytes(mt.ModelConfig(**bad))
    assert e.value.code == -1
    with pytest.raises(mt.MTError):
        mt.arena_bytes(mt.ModelConfig(**dict(CFGS["tiny"], n_heads=3)))
    with pytest.raises(mt.MTError):
        mt.arena_bytes(mt.ModelConfig(**dict(CFGS["tiny"], n_kv_heads=3)))
    with pytest.raises(mt.MTError):
        mt.tensor_offset(mt.ModelConfig(**CFGS["tiny"]), 5, 0, 0)


def test_adam_apply_rejects_bad_arguments(mt):
    cfg = mt.ModelConfig(**CFGS["tiny"])
    arena = mt.HostArena(mt.arena_bytes(cfg), pinned=False)
    with pytest.raises(mt.MTError):
        mt.adam_apply(cfg, arena, 0)  # step must be >= 1
    small = mt.HostArena(4096, pinned=False)
    with pytest.raises(mt.MTError):
        mt.adam_apply(cfg, small, 1)


# ------------------------------------------------------------------ fp32 master weights
@pytest.mark.parametrize("name", ["tiny", "gqa_ragged", "14b"])
def test_master_layout_matches_oracle(mt, name):
    cfg = mt.ModelConfig(**CFGS[name], flags=mt.FLAG_FP32_MASTER)
    ocfg = oracle.Config(**CFGS[name], fp32_master=True)
    lay = oracle.layout(ocfg)
    assert mt.arena_bytes(cfg) == lay["total"]
    for b, blk in enumerate(lay["blocks"]):
        assert mt.block_offset(cfg, b) == (blk["offset"], blk["bytes"])
        for si, sec in enumerate("WGMVP"):
            for ti, (tname, _) in enumerate(oracle.model.block_tensors(ocfg, b)):
                off, _, _, esz = mt.tensor_offset(cfg, b, si, ti)
                assert off == blk["sections"][sec]["tensors"][tname], (b, sec, tname)
                assert esz == (2 if sec in "WG" else 4)
    with pytest.raises(mt.MTError):  # no P section without the flag
        mt.tensor_offset(mt.ModelConfig(**CFGS[name]), 1, mt.SEC_P, 0)


def test_master_packing_bit_exact(mt):
    kw = CFGS["gqa_ragged"]
    cfg, ocfg = mt.ModelConfig(**kw, flags=mt.FLAG_FP32_MASTER), oracle.Config(**kw, fp32_master=True)
    arena = mt.HostArena(mt.arena_bytes(cfg), pinned=False)
    arena.array[:] = 0xAB
    mt.fill_synthetic(cfg, arena, synth, synth.WEIGHT_SEED)
    ref = oracle.pack_arena(ocfg, oracle.init_params(ocfg, synth, synth.WEIGHT_SEED))
    assert arena.array.tobytes() == ref.tobytes()


@pytest.mark.parametrize("step", [1, 3])
def test_master_host_adam_matches_oracle(mt, step):
    kw = CFGS["tiny"]
    cfg, ocfg = mt.ModelConfig(**kw, flags=mt.FLAG_FP32_MASTER), oracle.Config(**kw, fp32_master=True)
    arena = _random_arena(mt, cfg, ocfg, seed=10 + step)
    rng = np.random.default_rng(step)
    for blk in oracle.unpack_arena(ocfg, arena.array, "P"):  # masters off the bf16 grid
        for v in blk.values():
            v[...] = v + (rng.standard_normal(v.shape) * 1e-4).astype(np.float32)
    before = arena.array.copy()
    mt.adam_apply(cfg, arena, step)
    W0, G0, M0, V0, P0 = (oracle.unpack_arena(ocfg, before, s) for s in "WGMVP")
    W1, P1 = (oracle.unpack_arena(ocfg, arena.array, s) for s in "WP")
    for b in range(len(W0)):
        for k in W0[b]:
            w, _, _, p = oracle.adam_update(W0[b][k], G0[b][k], M0[b][k], V0[b][k], step, master=P0[b][k])
            # the master moves by at most ~lr; fp32 vs float64 arithmetic: a few fp32 ulp of the
            # master plus the update's own relative error (its m may cancel) times lr
            assert np.all(np.abs(P1[b][k] - p) <= 4 * 2.0 ** -24 * np.abs(p) + 1e-4 * 1e-3 + 1e-12), (b, k)
            # the stored weight is the bf16 rounding of the stored master, exactly
            np.testing.assert_array_equal(W1[b][k], oracle.float_to_bf16_bits(P1[b][k].astype(np.float64)))
            got, ref = oracle.bf16_bits_to_float(W1[b][k]), oracle.bf16_bits_to_float(w)
            assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-7), (b, k)


def test_master_host_adam_closed_form(mt):
    """The product's Adam with master weights on the constant-gradient case pinned in the oracle
    tests: w = 0.5, g = bf16(0.1), lr = 1e-4: w stays 0.5 for 9 steps and is 0.498046875 at
    step 10, the master then ~0.499; without master weights w stays 0.5."""
    kw = CFGS["tiny"]
    for flags, expect in ((mt.FLAG_FP32_MASTER, 0.498046875), (0, 0.5)):
        cfg = mt.ModelConfig(**kw, flags=flags)
        ocfg = oracle.Config(**kw, fp32_master=bool(flags))
        arena = mt.HostArena(mt.arena_bytes(cfg), pinned=False)
        arena.array[:] = 0
        W = oracle.unpack_arena(ocfg, arena.array, "W")
        G = oracle.unpack_arena(ocfg, arena.array, "G")
        W[1]["wq"][0, 0] = oracle.float_to_bf16_bits(np.array(0.5))
        G[1]["wq"][0, 0] = oracle.float_to_bf16_bits(np.array(0.1))
        if flags:
            mt.master_init(cfg, arena)
        for t in range(1, 11):
            mt.adam_apply(cfg, arena, t, lr=1e-4)
            w = float(oracle.bf16_bits_to_float(W[1]["wq"][0, :1])[0])
            assert w == (expect if t == 10 else 0.5), (flags, t, w)
        if flags:
            P = oracle.unpack_arena(ocfg, arena.array, "P")
            assert abs(float(P[1]["wq"][0, 0]) - 0.499) < 2e-6


def test_master_init_checks(mt):
    cfg = mt.ModelConfig(**CFGS["tiny"])
    arena = mt.HostArena(mt.arena_bytes(cfg), pinned=False)
    with pytest.raises(mt.MTError):  # no master section without the flag
        mt.master_init(cfg, arena)
    mcfg = mt.ModelConfig(**CFGS["tiny"], flags=mt.FLAG_FP32_MASTER)
    short = mt.HostArena(mt.arena_bytes(cfg), pinned=False)  # sized for 12 B/param
    with pytest.raises(mt.MTError):
        mt.master_init(mcfg, short)


@pytest.mark.parametrize("n_tiles,n_hb", [(1, 1), (32, 64), (32, 8), (32, 40), (1024, 32), (3, 17), (16, 4), (7, 33)])
def test_attention_block_order_covers_every_tile_once(mt, n_tiles, n_hb):
    """Every (tile, head pair) of a causal attention grid is taken by exactly one block, and
    inside each group of head pairs the ranks come heaviest first (non-decreasing in the block
    index), so the light tiles fill the end of the grid."""
    lib = mt._lib.load()
    rank, hb = ctypes.c_int(), ctypes.c_int()
    seen = set()
    last_rank = {}
    for lin in range(n_tiles * n_hb):
        assert lib.mtk_attn_block_slot(lin, n_tiles, n_hb, ctypes.byref(rank), ctypes.byref(hb)) == 0
        r, h = rank.value, hb.value
        assert 0 <= r < n_tiles and 0 <= h < n_hb
        seen.add((r, h))
        g = h // 16
        assert r >= last_rank.get(g, 0)
        last_rank[g] = r
    assert len(seen) == n_tiles * n_hb
    assert lib.mtk_attn_block_slot(n_tiles * n_hb, n_tiles, n_hb, ctypes.byref(rank), ctypes.byref(hb)) == -1  # MT_EINVAL
    assert lib.mtk_attn_block_slot(-1, n_tiles, n_hb, ctypes.byref(rank), ctypes.byref(hb)) == -1  # MT_EINVAL
    assert lib.mtk_attn_block_slot(0, n_tiles, n_hb, None, ctypes.byref(hb)) == -1  # MT_EINVAL
