"""The host page pool of the paged KV cache (spec_page_pool_*): pages come
from the free list in order, a sequence's mapped pages are a prefix of its
table row, release returns exactly the pages past the kept prefix (last
first), no page is ever mapped twice, and an exhausted pool refuses a
reservation without taking anything.  Host code only."""
import numpy as np
import pytest


@pytest.fixture(scope="module")
def sb():
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decoding_verification_pass_gb300 import binding
    return binding


def _pool(sb, n_pages, batch, max_pages):
    import ctypes
    h = ctypes.c_void_p()
    assert sb.lib().spec_page_pool_create(n_pages, batch, max_pages, ctypes.byref(h)) == sb.SPEC_OK
    return h.value


def _table(sb, h, batch, max_pages):
    ptr = sb.lib().spec_page_pool_table(h)
    return np.ctypeslib.as_array(ptr, shape=(batch * max_pages,)).reshape(batch, max_pages).copy()


def test_reserve_release_roundtrip(sb):
    L = sb.lib()
    h = _pool(sb, 10, 3, 5)
    assert L.spec_page_pool_reserve(h, 0, 130) == sb.SPEC_OK      # 3 pages
    assert L.spec_page_pool_reserve(h, 1, 64) == sb.SPEC_OK       # 1 page
    t = _table(sb, h, 3, 5)
    assert t[0, :3].tolist() == [0, 1, 2] and t[1, 0] == 3 and (t[0, 3:] == -1).all()
    assert L.spec_page_pool_free_pages(h) == 6
    assert L.spec_page_pool_reserve(h, 0, 100) == sb.SPEC_OK      # already covered
    assert L.spec_page_pool_free_pages(h) == 6
    assert L.spec_page_pool_release(h, 0, 65) == sb.SPEC_OK       # keep 2 pages: page 2 returns
    t = _table(sb, h, 3, 5)
    assert t[0].tolist() == [0, 1, -1, -1, -1]
    assert L.spec_page_pool_reserve(h, 2, 64) == sb.SPEC_OK       # takes the returned page
    assert _table(sb, h, 3, 5)[2, 0] == 2
    assert L.spec_page_pool_release(h, 0, 0) == sb.SPEC_OK
    assert L.spec_page_pool_release(h, 1, 0) == sb.SPEC_OK
    assert L.spec_page_pool_free_pages(h) == 9
    L.spec_page_pool_destroy(h)


def test_random_traffic_keeps_pages_unique(sb):
    L = sb.lib()
    rng = np.random.default_rng(3)
    B, P, NP = 8, 16, 60
    h = _pool(sb, NP, B, P)
    slots = [0] * B
    for _ in range(2000):
        b = int(rng.integers(0, B))
        if rng.random() < 0.6:
            want = slots[b] + int(rng.integers(1, 200))
            before = L.spec_page_pool_free_pages(h)
            r = L.spec_page_pool_reserve(h, b, want)
            if r == sb.SPEC_OK:
                slots[b] = max(slots[b], want)
            else:
                assert r == sb.SPEC_ESIZE and L.spec_page_pool_free_pages(h) == before
        else:
            keep = int(rng.integers(0, slots[b] + 1))
            assert L.spec_page_pool_release(h, b, keep) == sb.SPEC_OK
            slots[b] = keep
        t = _table(sb, h, B, P)
        used = t[t >= 0]
        assert len(set(used.tolist())) == used.size                  # no page mapped twice
        assert used.size + L.spec_page_pool_free_pages(h) == NP      # nothing lost
        for bb in range(B):
            n = -(-slots[bb] // 64)
            assert (t[bb, :n] >= 0).all() and (t[bb, n:] == -1).all()
    L.spec_page_pool_destroy(h)


def test_bad_arguments(sb):
    L = sb.lib()
    h = _pool(sb, 4, 2, 2)
    assert L.spec_page_pool_reserve(h, 2, 10) == sb.SPEC_EINVAL
    assert L.spec_page_pool_reserve(h, 0, 129) == sb.SPEC_ESIZE      # more than max_pages
    assert L.spec_page_pool_reserve(h, 0, -1) == sb.SPEC_EINVAL
    L.spec_page_pool_destroy(h)
