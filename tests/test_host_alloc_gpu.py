"""The arena allocator (mt_host_alloc / mt_host_free): page-locked, zero-filled, aligned to the
transparent-huge-page size when the kernel offers huge pages, and usable for asynchronous
copies in both directions and as a context's arena."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _thp_size():
    try:
        mode = open("/sys/kernel/mm/transparent_hugepage/enabled").read()
        size = int(open("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size").read())
    except (OSError, ValueError):
        return 0
    return 0 if "[never]" in mode else size


def _vma(ptr):
    """(start, end, AnonHugePages bytes) of the mapping holding ptr, from /proc/self/smaps."""
    cur = None
    for line in open("/proc/self/smaps"):
        head = line.split()
        if "-" in head[0] and len(head) >= 5:
            a, b = (int(x, 16) for x in head[0].split("-"))
            cur = (a, b) if a <= ptr < b else None
        elif cur and head[0] == "AnonHugePages:":
            return cur[0], cur[1], int(head[1]) * 1024
    return None


@pytest.fixture(scope="module")
def mt():
    from host_memory_streamed_stream_gb300 import _build

    _build.build()
    import host_memory_streamed_stream_gb300 as mt

    return mt


def test_arena_memory_is_pinned_zeroed_and_copies_both_ways(mt):
    torch.cuda.init()
    n = (3 << 29) + 4096  # 1.5 GiB and a bit: the last huge page is partly used
    a = mt.HostArena(n)
    try:
        hp = _thp_size()
        assert a.ptr % 4096 == 0
        if hp:
            assert a.ptr % hp == 0
            vma = _vma(a.ptr)
            assert vma is not None and vma[0] <= a.ptr and a.ptr + n <= vma[1]
            print(f"huge-page backed: {vma[2] / max(1, vma[1] - vma[0]):.3f} of the mapping")
            info = a.info()  # the allocator timed a copy of every huge page
            assert info is not None and info["huge_page_bytes"] == hp and info["huge_pages"] == 4
            assert 0 <= info["slow_found"] <= info["huge_pages"] and 0 <= info["replaced"] <= info["spare"]
            assert info["spare"] >= 8
            assert 0 < info["min_gbs"] <= info["median_gbs"]
            print("allocator:", info)
        idx = np.random.default_rng(0).integers(0, n, 4096)
        assert not a.array[idx].any() and not a.array[:4096].any() and not a.array[-4096:].any()
        h = torch.from_numpy(a.array)
        assert h.is_pinned()
        src = torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda")
        h.copy_(src, non_blocking=True)
        back = torch.empty_like(src)
        back.copy_(h, non_blocking=True)
        torch.cuda.synchronize()
        assert torch.equal(back, src)
    finally:
        a.free()


def test_arena_bound_to_a_context_after_allocation(mt):
    """A Trainer over an arena from the allocator binds it without registering it again."""
    cfg = mt.ModelConfig(n_layers=1, hidden=256, n_heads=4, n_kv_heads=4, ffn=512, vocab=512, seq=64, batch=1)
    a = mt.HostArena(mt.arena_bytes(cfg))
    try:
        import synth

        mt.fill_synthetic(cfg, a, synth, synth.WEIGHT_SEED)
        with mt.Trainer(cfg, arena=a) as tr:
            loss = tr.step(synth.tokens(cfg.tokens, cfg.vocab), synth.labels(cfg.tokens, cfg.vocab))
            assert np.isfinite(loss) and abs(loss - np.log(cfg.vocab)) < 0.5
    finally:
        a.free()
