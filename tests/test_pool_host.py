"""The page ledger and the native page pool (host code of the C library, no
GPU): page bytes from the 9-byte NVFP4 block, the equal-memory capacity of a
precision map pinned to the pages' 44 -> 70 figure, and the pool's
all-or-nothing allocation and checked release."""
import pytest

from conftest import read_golden


@pytest.fixture(scope="module")
def nv():
    import nvfp4_quantized_paged_gb300 as nv
    return nv


def test_page_bytes_follow_the_block_ledger(nv):
    # 16 values: 9 bytes in NVFP4 (8 code bytes + 1 scale byte), 16 in FP8; K and V
    assert nv.nvkv_cache_page_bytes(nv.PREC_NVFP4, 64, 8, 128) == 64 * 8 * 2 * (128 // 16) * 9
    assert nv.nvkv_cache_page_bytes(nv.PREC_FP8, 64, 8, 128) == 64 * 8 * 2 * 128
    assert nv.nvkv_cache_page_bytes(nv.PREC_NVFP4, 16, 2, 100) == 0  # head_dim not a multiple of 16
    assert nv.nvkv_cache_page_bytes(7, 16, 2, 128) == 0


def test_equal_memory_capacity_matches_the_pages(nv):
    want = {k: int(v) for k, v in read_golden("capacity.txt")}
    L, P, layers, Hkv = 4096, 64, 28, 8
    pages_per_seq = L // P
    fp8_map = [nv.PREC_FP8] * layers
    mixed_map = [nv.PREC_FP8 if l in (0, 25, 26, 27) else nv.PREC_NVFP4 for l in range(layers)]
    budget = want["fp8_sequences"] * pages_per_seq * layers * nv.nvkv_cache_page_bytes(nv.PREC_FP8, P, Hkv)
    cap = {}
    for name, m in (("fp8_sequences", fp8_map), ("mixed_sequences", mixed_map)):
        pool = nv.PagePool(nv.nvkv_pool_pages_for_budget(budget, m, P, Hkv))
        n = 0
        while pool.alloc(pages_per_seq) is not None:
            n += 1
        cap[name] = n
        assert pool.num_free < pages_per_seq
    assert cap == want
    # all-NVFP4: the ideal 16/9 = 1.78x of the ledger, floored to whole sequences
    nv_pages = nv.nvkv_pool_pages_for_budget(budget, [nv.PREC_NVFP4] * layers, P, Hkv)
    assert nv_pages == (budget // (layers * nv.nvkv_cache_page_bytes(nv.PREC_NVFP4, P, Hkv)))
    assert nv_pages // pages_per_seq == (44 * 16) // 9


def test_pool_allocation_and_release(nv):
    pool = nv.PagePool(6)
    a = pool.alloc(4)
    assert a == [0, 1, 2, 3] and pool.num_free == 2
    assert pool.alloc(3) is None and pool.num_free == 2  # all or nothing
    pool.release([2, 0])
    assert pool.num_free == 4
    b = pool.alloc(4)
    assert sorted(b) == [0, 2, 4, 5] and pool.num_free == 0
    with pytest.raises(nv.NvkvError):
        pool.release([1, 1])  # listed twice: nothing released
    assert pool.num_free == 0
    with pytest.raises(nv.NvkvError):
        pool.release([6])  # out of range
    pool.release([1, 3])
    with pytest.raises(nv.NvkvError):
        pool.release([3])  # not held any more
    assert pool.num_free == 2
    assert pool.alloc(0) == []
    pool.close()
