"""The expert cache's replacement policy (moe_cache_plan: the decisions of
moe_cache_ensure without CUDA work), checked on CPU against hand-traced LRU
sequences: empty slots fill first in slot order, then the least recently listed
slot that holds no currently listed expert is evicted (the lower slot on ties)."""
import ctypes as C

import pytest

import moe_expert_layer_03_gb300 as moe


@pytest.fixture()
def cache():
    L = moe.lib()
    pool = moe.MoePool(8, 4, 256, 512, 1, 0x10000000, 1 << 20, 0x20000000)   # never dereferenced
    h = C.c_void_p()
    assert L.moe_cache_create(C.byref(pool), C.c_void_p(0x30000000), 1, C.byref(h)) == 0   # DMA copies
    yield L, h
    L.moe_cache_destroy(h)


def plan(L, h, experts):
    n = 4
    ex = (C.c_int32 * max(1, len(experts)))(*experts)
    le, ls, nl = (C.c_int32 * n)(), (C.c_int32 * n)(), C.c_int(0)
    st = L.moe_cache_plan(h, C.cast(ex, C.c_void_p), len(experts), C.cast(le, C.c_void_p),
                          C.cast(ls, C.c_void_p), C.byref(nl))
    return st, [(le[i], ls[i]) for i in range(nl.value)]


def test_lru_sequence(cache):
    L, h = cache
    assert plan(L, h, [3, 1]) == (0, [(3, 0), (1, 1)])    # tick 1: empty slots in order
    assert plan(L, h, [1, 5]) == (0, [(5, 2)])            # tick 2: 1 hits
    assert plan(L, h, [7, 2]) == (0, [(7, 3), (2, 0)])    # tick 3: last empty slot; evict 3 (tick 1)
    assert plan(L, h, [5]) == (0, [])                     # tick 4: hit
    # tick 5: slots 0 (2, t3), 1 (1, t2), 2 (5, t4), 3 (7, t3): 4 evicts 1; 6 then evicts
    # slot 0 (t3, ties with slot 3 and the lower slot goes)
    assert plan(L, h, [4, 6]) == (0, [(4, 1), (6, 0)])
    # a listed expert is never evicted, even when it is the least recently used
    assert plan(L, h, [7, 0, 1, 5]) == (0, [(0, 0), (1, 1)])   # slots 3, 2 hold 7, 5 -> hits
    c = moe.CacheCounters()
    assert L.moe_cache_stats(h, C.byref(c)) == 0
    assert (c.hits, c.misses, c.bytes_copied) == (4, 9, 9 << 20)   # 2+1+2+0+2+2 loads


def test_rejections(cache):
    L, h = cache
    assert plan(L, h, [0, 1, 2, 3, 4])[0] == 2    # more experts than slots
    assert plan(L, h, [1, 1])[0] == 1             # duplicate
    assert plan(L, h, [8])[0] == 1                # outside [0, E)
    assert plan(L, h, [-1])[0] == 1
    assert plan(L, h, [])[0] == 0                 # nothing listed: nothing to do
