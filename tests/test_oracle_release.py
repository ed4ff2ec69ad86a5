"""Oracle pins for the page lifecycle: release, reallocation and the tag
check of append ("Smaller, faster, safer: running Kimi and GLM at scale",
section "Protecting a shared KV cache": a page's tag changes whenever the page
is reallocated, and a request whose recorded tags no longer match is aborted).

The expected states below are worked out by hand from the rules the oracle
states: pops from free_list[free_head], tag += 1 per pop, release pushes the
released pages back below free_head in (request, page) order."""
import numpy as np
import pytest

import oracle

P = 4


def _pool():
    return oracle.Pool(8, P, 1, 16, 16, dtype=0, layout=0,
                       tags=[10, 20, 30, 40, 50, 60, 70, 80],
                       free_list=[5, 2, 7, 0, 3, 6, 1, 4])


def _state(B=3, mp=4):
    return (np.full((B, mp), -1, np.int32), np.zeros((B, mp), np.uint32),
            np.zeros(B, np.int32))


def _ind(ns):
    return np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)


def test_release_then_reallocate_by_hand():
    pool = _pool()
    pt, et, sl = _state()
    assert oracle.alloc(pool, _ind([5, 3, 8]), 8, pt, et, sl) == (0, 3)
    assert pt.tolist() == [[5, 2, -1, -1], [7, -1, -1, -1], [0, 3, -1, -1]]
    assert et.tolist() == [[61, 31, 0, 0], [81, 0, 0, 0], [11, 41, 0, 0]]
    assert int(pool.free_head[0]) == 5 and sl.tolist() == [5, 3, 8]
    old_pt0, old_et0 = pt[0:1].copy(), et[0:1].copy()

    assert oracle.release(pool, pt, et, sl, np.array([1, 0, 1], np.uint8)) == 0
    assert int(pool.free_head[0]) == 1
    assert pool.free_list[1:5].tolist() == [5, 2, 0, 3]   # request 0's pages, then 2's
    assert pt.tolist() == [[-1] * 4, [7, -1, -1, -1], [-1] * 4]
    assert et.tolist() == [[0] * 4, [81, 0, 0, 0], [0] * 4]
    assert sl.tolist() == [0, 3, 0]
    assert pool.tags.tolist() == [11, 20, 31, 41, 50, 61, 70, 81]  # release leaves tags

    # request 0 takes one page, request 1 fills its page 0 (tag still 81)
    # and takes one more: the released pages come back in order, tags bumped
    assert oracle.alloc(pool, _ind([4, 2, 0]), 4, pt, et, sl) == (0, 3)
    assert pt.tolist() == [[5, -1, -1, -1], [7, 2, -1, -1], [-1] * 4]
    assert et.tolist() == [[62, 0, 0, 0], [81, 32, 0, 0], [0] * 4]
    assert int(pool.free_head[0]) == 3 and sl.tolist() == [4, 5, 0]

    # the mapping request 0 recorded before its release is now stale
    m = oracle.verify(8, P, pool.tags, old_pt0, old_et0, np.array([5], np.int32))
    assert m.tolist() == [1]
    assert oracle.verify(8, P, pool.tags, pt, et, sl).tolist() == [0, 0, 0]


def test_append_refuses_a_reallocated_partial_page():
    pool = _pool()
    pt, et, sl = _state()
    oracle.alloc(pool, _ind([5, 3, 8]), 8, pt, et, sl)
    snap = (pt.copy(), et.copy(), sl.copy(), pool.tags.copy(), int(pool.free_head[0]))
    pool.tags[7] += 1  # request 1's partly filled page 7 was handed out elsewhere
    st, stop = oracle.alloc(pool, _ind([0, 1, 4]), 4, pt, et, sl)
    assert (st, stop) == (oracle.ERR_TAG_MISMATCH, 1)
    assert np.array_equal(pt, snap[0]) and np.array_equal(et, snap[1])
    assert np.array_equal(sl, snap[2]) and int(pool.free_head[0]) == snap[4]
    # a full last page is not written again, so no check applies: request 2
    # (8 rows = 2 full pages) appends without touching page 3
    pool.tags[3] += 5
    st, stop = oracle.alloc(pool, _ind([0, 0, 4]), 4, pt, et, sl)
    assert (st, stop) == (0, 3) and pt[2].tolist() == [0, 3, 6, -1]
    # an out-of-range id in the partly filled slot
    pt[0, 1] = 99
    st, stop = oracle.alloc(pool, _ind([1, 0, 0]), 1, pt, et, sl)
    assert (st, stop) == (oracle.ERR_BAD_PAGE_ID, 0)


def test_append_sees_a_partial_page_popped_earlier_in_the_same_call():
    """Requests are served in order: a partly filled page that an earlier
    request of the same call pops has its tag bumped before the later
    request's check, which then fails."""
    pool = _pool()
    pt, et, sl = _state()
    oracle.alloc(pool, _ind([5, 3, 8]), 8, pt, et, sl)
    # request 1's partly filled page 7 (3 of 4 slots) is listed free again,
    # at the top of the free list (free_head = 5)
    pool.free_list[5] = 7
    st, stop = oracle.alloc(pool, _ind([4, 1, 0]), 4, pt, et, sl)
    # request 0 (5 -> 9 rows) checks its page 2 (tag 31: ok) and pops page 7
    # (tag 81 -> 82); request 1 then finds tag 82 against its recorded 81
    assert (st, stop) == (oracle.ERR_TAG_MISMATCH, 1)
    assert pt.tolist() == [[5, 2, 7, -1], [7, -1, -1, -1], [0, 3, -1, -1]]
    assert et.tolist() == [[61, 31, 82, 0], [81, 0, 0, 0], [11, 41, 0, 0]]
    assert sl.tolist() == [9, 3, 8] and int(pool.free_head[0]) == 6
    assert int(pool.tags[7]) == 82


def test_release_failures_change_nothing():
    pool = _pool()
    pt, et, sl = _state()
    oracle.alloc(pool, _ind([5, 3, 8]), 8, pt, et, sl)
    snap = (pt.copy(), et.copy(), sl.copy(), pool.free_list.copy(), int(pool.free_head[0]))

    def same():
        return (np.array_equal(pt, snap[0]) and np.array_equal(et, snap[1]) and
                np.array_equal(sl, snap[2]) and np.array_equal(pool.free_list, snap[3]) and
                int(pool.free_head[0]) == snap[4])

    pool.free_head[0] = 4  # only 4 pages handed out, the requests own 5
    assert oracle.release(pool, pt, et, sl) == oracle.ERR_INVALID_ARG
    pool.free_head[0] = snap[4]
    assert same()
    sl[1] = -1
    assert oracle.release(pool, pt, et, sl, np.array([0, 1, 0], np.uint8)) == oracle.ERR_INVALID_ARG
    sl[1] = 17  # 5 pages > max_pages
    assert oracle.release(pool, pt, et, sl, np.array([0, 1, 0], np.uint8)) == oracle.ERR_INVALID_ARG
    sl[1] = snap[2][1]
    assert same()
    # releasing nobody, or a request that owns nothing, is a no-op
    assert oracle.release(pool, pt, et, sl, np.zeros(3, np.uint8)) == 0 and same()


def test_release_everything_returns_the_pool():
    pool = _pool()
    pt, et, sl = _state()
    oracle.alloc(pool, _ind([5, 3, 8]), 8, pt, et, sl)
    assert oracle.release(pool, pt, et, sl) == 0  # NULL mask: every request
    assert int(pool.free_head[0]) == 0
    assert sorted(pool.free_list[:5].tolist()) == [0, 2, 3, 5, 7]
    assert (pt == -1).all() and (et == 0).all() and (sl == 0).all()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_lifecycle_invariants_random(seed):
    """Random append / release rounds: every page is owned by exactly one
    request or is free; each tag grew by the number of times the page was
    popped; verify never aborts a live request."""
    rng = np.random.default_rng(seed)
    npg, B, mp = 64, 6, 16
    tags0 = rng.integers(0, 2 ** 32, npg, dtype=np.uint64).astype(np.uint32)
    pool = oracle.Pool(npg, P, 1, 16, 16, tags=tags0, free_list=rng.permutation(npg))
    pt, et, sl = _state(B, mp)
    pops = np.zeros(npg, np.int64)
    for _ in range(40):
        if rng.random() < 0.6:
            ns = rng.integers(0, 9, B)
            head0 = int(pool.free_head[0])
            st, stop = oracle.alloc(pool, _ind(ns), 8, pt, et, sl)
            for p in pool.free_list[head0:int(pool.free_head[0])]:
                pops[p] += 1
        else:
            st = oracle.release(pool, pt, et, sl, (rng.random(B) < 0.4).astype(np.uint8))
            assert st == 0
        owned = [int(pt[r, j]) for r in range(B) for j in range(-(-int(sl[r]) // P))]
        free = pool.free_list[int(pool.free_head[0]):].tolist()
        assert sorted(owned + free) == list(range(npg))
        assert np.array_equal(pool.tags, (tags0.astype(np.int64) + pops).astype(np.uint32))
        assert not oracle.verify(npg, P, pool.tags, pt, et, sl).any()
