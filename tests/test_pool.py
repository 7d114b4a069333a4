"""The shared-pool allocator (host code in libcarat.so, no GPU needed).

Rings are aligned runs of pages, single pages fill blocks that pages already
broke up before taking whole blocks, allocation is all-or-nothing, and a
random sequence of operations never hands out a page twice."""
import os
import random

import pytest


@pytest.fixture(scope="module")
def carat():
    from sliding_window_gqa_ring_gb300 import build, carat as c
    if not os.path.exists(c.LIBRARY):
        build.build()
    c.library()
    return c


def test_rings_are_aligned_blocks_from_the_bottom(carat):
    pool = carat.Pool(64, 8)
    assert [pool.alloc_ring() for _ in range(3)] == [0, 1, 2]
    assert pool.stats() == {"free_pages": 40, "whole_free_blocks": 5, "rings": 3, "pages": 0}


def test_pages_fill_broken_blocks_first_from_the_top(carat):
    pool = carat.Pool(64, 8)
    a = pool.alloc_pages(3)
    assert a == [56, 57, 58]                   # top block broken up
    b = pool.alloc_pages(6)
    assert b == [59, 60, 61, 62, 63, 48]       # finish it, then the next block down
    assert pool.stats()["whole_free_blocks"] == 6
    assert pool.alloc_ring() == 0               # rings still find whole blocks


def test_tail_pages_past_the_last_block_go_first(carat):
    pool = carat.Pool(20, 8)                    # 2 blocks + 4 tail pages
    assert pool.alloc_pages(5) == [16, 17, 18, 19, 8]   # then the highest whole block
    assert pool.alloc_ring() == 0
    assert pool.alloc_ring() == -1              # block 1 is broken up


def test_all_or_nothing(carat):
    pool = carat.Pool(32, 8)
    assert pool.alloc_ring() == 0
    before = pool.stats()
    assert pool.alloc_pages(25) is None         # only 24 free
    assert pool.stats() == before
    got = pool.alloc_pages(24)
    assert sorted(got) == list(range(8, 32))
    assert pool.alloc_ring() == -1


def test_frees_are_checked_and_atomic(carat):
    pool = carat.Pool(16, 4)
    r = pool.alloc_ring()
    pages = pool.alloc_pages(4)
    assert not pool.free_pages([pages[0], pages[0]])      # listed twice
    assert not pool.free_pages([pages[1], 0])             # page 0 belongs to a ring
    assert pool.stats()["pages"] == 4                     # nothing was freed
    assert pool.free_pages(pages)
    assert not pool.free_ring(r + 1)
    assert pool.free_ring(r)
    assert not pool.free_ring(r)
    assert pool.stats() == {"free_pages": 16, "whole_free_blocks": 4, "rings": 0, "pages": 0}


def test_random_operations_never_overlap(carat):
    rng = random.Random(5)
    npages, ppr = 203, 8
    pool = carat.Pool(npages, ppr)
    rings, pages = set(), set()
    for _ in range(3000):
        op = rng.random()
        if op < 0.3:
            r = pool.alloc_ring()
            if r >= 0:
                assert r not in rings
                rings.add(r)
        elif op < 0.6:
            got = pool.alloc_pages(rng.randint(1, 12))
            if got is not None:
                assert not pages & set(got)
                pages |= set(got)
        elif op < 0.8 and rings:
            r = rng.choice(sorted(rings))
            assert pool.free_ring(r)
            rings.discard(r)
        elif pages:
            some = rng.sample(sorted(pages), min(len(pages), rng.randint(1, 6)))
            assert pool.free_pages(some)
            pages -= set(some)
        ring_pages = {r * ppr + i for r in rings for i in range(ppr)}
        assert not ring_pages & pages
        assert all(0 <= p < npages for p in pages)
        st = pool.stats()
        assert st["rings"] == len(rings) and st["pages"] == len(pages)
        assert st["free_pages"] == npages - len(pages) - len(ring_pages)


def test_bad_pool_arguments(carat):
    with pytest.raises(carat.CaratError):
        carat.Pool(0, 8)
    with pytest.raises(carat.CaratError):
        carat.Pool(8, 0)
