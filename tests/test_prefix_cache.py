"""The KV-only prefix-sharing page allocator (host side, no GPU).

"Accelerating GLM-5.3-Flash on H200", section 2 "KV-only decode
RadixCache": N requests with a shared prefix of Lp tokens and private
suffixes of Ls tokens occupy Lp + N·Ls slots.  With pages as the unit of
sharing, the prefix counts in whole pages.  The allocator is checked against
that formula, against the decode workload's layout (81,792 slots), against a
plain model of "one page per distinct whole-page prefix", and for its
reference counting, eviction order and failure behaviour.
"""
import random
import threading

import numpy as np
import pytest

import dsa_sparse_mla_topk_gb300 as dsa
from dsa_sparse_mla_topk_gb300 import build as dsa_build
from dsa_sparse_mla_topk_gb300 import workloads as wl


@pytest.fixture(scope="module", autouse=True)
def _lib():
    dsa_build.build()
    dsa.load_library()


def _tokens(rng, n):
    return rng.integers(0, 50000, size=n, dtype=np.int32)


def test_decode_workload_layout_is_reproduced():
    """128 requests, 65,470 shared tokens + 66 private, page 64: 1022 shared
    pages and 2 private pages per request, 81,792 slots, as the input
    generator lays out the decode workload."""
    w = wl.WORKLOADS["decode_64k_prefix99.9"]
    P = w.page_size
    rng = np.random.default_rng(0)
    prefix = _tokens(rng, w.shared_prefix)
    cache = dsa.PrefixCache(P, wl.slot_count(w) // P)
    tables = []
    for r in range(w.num_req):
        bt, shared = cache.acquire(np.concatenate([prefix, _tokens(rng, w.ctx - w.shared_prefix)]))
        assert len(bt) == w.ctx // P
        assert shared == (0 if r == 0 else w.shared_prefix // P)
        tables.append(bt)
    referenced, cached, free = cache.stats()
    assert referenced * P == wl.slot_count(w) == 81_792 and free == 0
    first = np.stack([t[:1022] for t in tables])
    assert (first == first[0]).all()
    private = np.concatenate([t[1022:] for t in tables])
    assert len(np.unique(private)) == len(private) == 2 * w.num_req
    assert not set(private) & set(first[0])


@pytest.mark.parametrize("lp_pages,ls,n", [(4, 10, 7), (16, 64, 5), (0, 33, 3)])
def test_slots_follow_lp_plus_n_ls(lp_pages, ls, n):
    P = 16
    rng = np.random.default_rng(lp_pages + ls)
    prefix = _tokens(rng, lp_pages * P)
    cache = dsa.PrefixCache(P, 1000)
    for _ in range(n):
        cache.acquire(np.concatenate([prefix, _tokens(rng, ls)]))
    referenced, _, _ = cache.stats()
    assert referenced * P == lp_pages * P + n * (-(-ls // P)) * P


def test_random_requests_match_a_model_of_distinct_page_prefixes():
    """Requests built from a few documents cut at random points: the cache
    holds exactly one page per distinct whole-page prefix, plus one private
    page per request with a partial last page; equal prefixes get equal ids."""
    P = 8
    rng = np.random.default_rng(3)
    docs = [_tokens(rng, 400) for _ in range(4)]
    cache = dsa.PrefixCache(P, 10_000)
    prefixes = {}
    partial = 0
    for _ in range(60):
        d = docs[rng.integers(len(docs))]
        n = int(rng.integers(1, 400))
        t = d[:n].copy()
        if rng.random() < 0.3:  # a private continuation
            t = np.concatenate([t, _tokens(rng, int(rng.integers(1, 40)))])
        bt, shared = cache.acquire(t)
        for p in range(len(t) // P):
            key = t[: (p + 1) * P].tobytes()
            if p < shared:
                assert prefixes[key] == bt[p]
            prefixes.setdefault(key, bt[p])
            assert prefixes[key] == bt[p]
        partial += len(t) % P != 0
    referenced, cached, free = cache.stats()
    assert cached == len(prefixes)
    assert referenced == len(prefixes) + partial
    assert free == 10_000 - referenced


def test_release_keeps_pages_cached_for_reuse():
    P = 4
    rng = np.random.default_rng(4)
    t = _tokens(rng, 22)
    cache = dsa.PrefixCache(P, 64)
    bt, shared = cache.acquire(t)
    assert shared == 0 and cache.stats() == (6, 5, 58)
    cache.release(bt)
    assert cache.stats() == (0, 5, 59)           # the partial page is free again
    bt2, shared2 = cache.acquire(t)
    assert shared2 == 5 and (bt2[:5] == bt[:5]).all()
    with pytest.raises(dsa.DsaError):
        cache.release(np.array([60], dtype=np.int32))  # a free page
    cache.release(bt2)


def test_eviction_takes_least_recently_used_unreferenced_leaves():
    P = 4
    rng = np.random.default_rng(5)
    a, b, c = _tokens(rng, 16), _tokens(rng, 16), _tokens(rng, 24)
    cache = dsa.PrefixCache(P, 10)
    bt_a, _ = cache.acquire(a)
    bt_b, _ = cache.acquire(b)
    cache.release(bt_a)                          # a released first: older
    cache.release(bt_b)
    assert cache.stats() == (0, 8, 2)
    bt_c, _ = cache.acquire(c)                   # 6 pages: 2 free + 4 evicted, all of a's
    assert sorted(set(bt_c) - {8, 9}) == sorted(bt_a)
    _, shared_b = cache.acquire(b)
    assert shared_b == 4                         # b survived
    cache.release(bt_c)                          # c's leaves become evictable
    bt_a2, shared_a = cache.acquire(a[:8])
    assert shared_a == 0                         # a's pages were evicted
    assert set(bt_a2) <= set(bt_c[-2:])          # the 2 deepest of c's pages made room


def test_out_of_pages_changes_nothing():
    P = 4
    rng = np.random.default_rng(6)
    cache = dsa.PrefixCache(P, 6)
    cache.acquire(_tokens(rng, 20))               # 5 pages, referenced
    before = cache.stats()
    with pytest.raises(dsa.DsaError) as e:
        cache.acquire(_tokens(rng, 9))            # needs 3, only 1 free, nothing evictable
    assert e.value.status == 5
    assert cache.stats() == before


def test_concurrent_acquire_and_release_keep_the_counts():
    P = 8
    cache = dsa.PrefixCache(P, 4096)
    prefix = np.arange(64, dtype=np.int32)
    cache.release(cache.acquire(prefix)[0])      # the prefix is cached before the threads start

    def worker(seed):
        rng = random.Random(seed)
        for _ in range(200):
            t = np.concatenate([prefix, np.array([rng.randrange(10**6) for _ in range(rng.randrange(1, 30))],
                                                 dtype=np.int32)])
            bt, shared = cache.acquire(t)
            assert shared == 8
            cache.release(bt)

    threads = [threading.Thread(target=worker, args=(s,)) for s in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    referenced, cached, free = cache.stats()
    assert referenced == 0 and free == 4096 - cached
