"""Pin the oracle's packed-block layout to the written rule (4 KB alignment, order, sizes)."""
import numpy as np

import oracle
import synth
from oracle import model as om

CFGS = {
    "tiny": oracle.Config(2, 256, 4, 4, 1024, 1024, 128, 2),
    "1.3b": oracle.Config(24, 2048, 16, 16, 5504, 32000, 2048, 4),
    "7b": oracle.Config(32, 4096, 32, 32, 11008, 32000, 4096, 2),
    "14b": oracle.Config(48, 5120, 40, 8, 13824, 152064, 4096, 1),
}


def test_alignment_and_order():
    for cfg in CFGS.values():
        lay = om.layout(cfg)
        prev_end = 0
        for b, blk in enumerate(lay["blocks"]):
            assert blk["offset"] == prev_end and blk["offset"] % 4096 == 0
            secs = blk["sections"]
            assert list(secs) == ["W", "G", "M", "V"]
            end = blk["offset"]
            for sec, esz in (("W", 2), ("G", 2), ("M", 4), ("V", 4)):
                s = secs[sec]
                assert s["offset"] == end and s["offset"] % 4096 == 0
                t_end = s["offset"]
                for name, shape in om.block_tensors(cfg, b):
                    o = s["tensors"][name]
                    assert o % 4096 == 0 and o == t_end
                    n = int(np.prod(shape)) * esz
                    t_end = o + (n + 4095) // 4096 * 4096
                assert t_end == s["offset"] + s["bytes"]
                end = t_end
            assert end == blk["offset"] + blk["bytes"]
            prev_end = end
        assert lay["total"] == prev_end


def test_total_bytes_closed_form():
    """12 bytes per parameter (2 W + 2 G + 4 M + 4 V) up to 4 KB padding per tensor."""
    for cfg in CFGS.values():
        h, f, V, L = cfg.hidden, cfg.ffn, cfg.vocab, cfg.n_layers
        qd = cfg.n_heads * cfg.head_dim
        kvd = cfg.n_kv_heads * cfg.head_dim
        per_layer = 2 * h + 2 * qd * h + 2 * kvd * h + 3 * f * h
        total = V * h + L * per_layer + h + V * h
        lay = om.layout(cfg)
        ntensors = 1 + 9 * L + 2
        assert 12 * total <= lay["total"] <= 12 * total + 4 * ntensors * 4096
    # the 7B model is 6.74 B parameters (80.9 GB at 12 B/param)
    cfg = CFGS["7b"]
    assert abs(om.layout(cfg)["total"] / 12 / 1e9 - 6.738) < 0.01


def test_pack_then_unpack_roundtrip():
    cfg = CFGS["tiny"]
    W = oracle.init_params(cfg, synth, synth.WEIGHT_SEED)
    arena = oracle.pack_arena(cfg, W)
    back = oracle.unpack_arena(cfg, arena, "W")
    for b in range(cfg.n_layers + 2):
        for k in W[b]:
            np.testing.assert_array_equal(back[b][k], W[b][k])
    for sec in ("G", "M", "V"):
        for blk in oracle.unpack_arena(cfg, arena, sec):
            for v in blk.values():
                assert not np.any(v)



def test_master_section_layout():
    """With float32 master weights a fifth section P (4 bytes/element) follows V: 16 bytes per
    parameter up to the 4 KB padding, every offset 4096-aligned, W/G/M/V where they were within
    each block's first four sections."""
    import dataclasses
    for cfg in CFGS.values():
        mcfg = dataclasses.replace(cfg, fp32_master=True)
        lay, mlay = om.layout(cfg), om.layout(mcfg)
        for b, (blk, mblk) in enumerate(zip(lay["blocks"], mlay["blocks"])):
            assert list(mblk["sections"]) == ["W", "G", "M", "V", "P"]
            base = mblk["offset"] - blk["offset"]
            for sec in "WGMV":
                for name, o in blk["sections"][sec]["tensors"].items():
                    assert mblk["sections"][sec]["tensors"][name] == o + base
            P = mblk["sections"]["P"]
            assert P["offset"] == mblk["sections"]["V"]["offset"] + mblk["sections"]["V"]["bytes"]
            assert P["bytes"] == mblk["sections"]["V"]["bytes"]  # same element size, same tensors
            assert all(o % 4096 == 0 for o in P["tensors"].values())
            assert mblk["offset"] + mblk["bytes"] == P["offset"] + P["bytes"]
        h, f, V, L = cfg.hidden, cfg.ffn, cfg.vocab, cfg.n_layers
        qd, kvd = cfg.n_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
        total = V * h + L * (2 * h + 2 * qd * h + 2 * kvd * h + 3 * f * h) + h + V * h
        ntensors = 1 + 9 * L + 2
        assert 16 * total <= mlay["total"] <= 16 * total + 5 * ntensors * 4096


def test_master_pack_holds_the_weights_as_float32():
    import dataclasses
    cfg = dataclasses.replace(CFGS["tiny"], fp32_master=True)
    W = oracle.init_params(cfg, synth, synth.WEIGHT_SEED)
    arena = oracle.pack_arena(cfg, W)
    P = oracle.unpack_arena(cfg, arena, "P")
    for b in range(cfg.n_layers + 2):
        for k in W[b]:
            np.testing.assert_array_equal(P[b][k], oracle.bf16_bits_to_float(W[b][k]).astype(np.float32))
