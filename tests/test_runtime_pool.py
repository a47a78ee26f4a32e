"""The host-side admission runtime (shared-affix registry and private-page allocator) on the CPU.

Source: "Affix Cache for Diffusion Large Language Models", Sec. 4.1-4.2: each common affix is
stored once in the shared region and reused by later compatible requests; every request gets
private slots for its anchors and own positions, and admission records them before the online
loop.  These checks are exact: no two live allocations overlap, references are counted,
released slots are reused, and exhaustion is reported, not hidden.
"""
import threading

import pytest

import affix_kv_cache_gb300 as ac
from affix_kv_cache_gb300 import _lib


def test_registry_reuses_and_refcounts_affixes():
    p = ac.Pool(num_slots=10_000, private_begin=4096, page_slots=256)
    base, created = p.register_affix(0xABC, 1024)
    assert created and base == 0
    again, created2 = p.register_affix(0xABC, 1024)
    assert again == base and not created2
    other, created3 = p.register_affix(0xDEF, 2048)
    assert created3 and other == 1024                   # first fit, no overlap
    assert p.stats()["free_shared"] == 4096 - 3072
    p.release_affix(0xABC)
    assert p.stats()["affixes"] == 2                    # one reference left
    p.release_affix(0xABC)
    assert p.stats()["affixes"] == 1 and p.stats()["free_shared"] == 4096 - 2048
    b3, c3 = p.register_affix(0x123, 512)               # reuses the freed run
    assert c3 and b3 == 0
    with pytest.raises(ac.AcacheError) as e:
        p.register_affix(0xDEF, 100)                    # same key, other length
    assert e.value.status == _lib.ACACHE_ERR_INVALID_ARG
    with pytest.raises(ac.AcacheError) as e:
        p.register_affix(0x999, 4096)                   # does not fit
    assert e.value.status == _lib.ACACHE_ERR_WORKSPACE
    p.release_affix(0x123)
    p.release_affix(0xDEF)
    assert p.stats()["free_shared"] == 4096             # runs coalesced back into one
    assert p.register_affix(0x777, 4096) == (0, True)


def test_private_pages_are_disjoint_and_recycled():
    # 16 requests of 1204 rows take 5 pages of 256 slots each: 80 pages, plus a partial page
    p = ac.Pool(num_slots=4096 + 80 * 256 + 100, private_begin=4096, page_slots=256)
    pages = 80
    assert p.stats()["free_private"] == pages * 256
    seen, ids = set(), []
    for r in range(16):
        slots, rid = p.alloc_private(1204)
        s = slots.tolist()
        assert len(set(s)) == 1204 and not (set(s) & seen)
        assert all(4096 <= x < 4096 + pages * 256 for x in s)
        seen |= set(s)
        ids.append(rid)
    assert p.stats()["requests"] == 16
    with pytest.raises(ac.AcacheError):
        p.alloc_private(1)                              # every whole page is taken
    p.free_private(ids[3])
    slots, rid = p.alloc_private(1204)
    assert set(slots.tolist()) <= seen                  # the freed pages come back
    with pytest.raises(ac.AcacheError):
        p.free_private(ids[3])                          # already freed
    for r in ids[:3] + ids[4:] + [rid]:
        p.free_private(r)
    assert p.stats()["free_private"] == pages * 256 and p.stats()["requests"] == 0


def test_zero_row_request_and_bad_arguments():
    p = ac.Pool(num_slots=1000, private_begin=0, page_slots=100)
    slots, rid = p.alloc_private(0)
    assert slots.numel() == 0
    p.free_private(rid)
    with pytest.raises(ac.AcacheError):
        p.register_affix(1, 1)                           # no shared region at all
    with pytest.raises(ac.AcacheError):
        ac.Pool(num_slots=10, private_begin=11, page_slots=4)
    with pytest.raises(ac.AcacheError):
        ac.Pool(num_slots=10, private_begin=0, page_slots=0)


def test_concurrent_admissions_never_share_a_slot():
    p = ac.Pool(num_slots=64 * 1000, private_begin=0, page_slots=64)
    got, lock = [], threading.Lock()

    def worker():
        for _ in range(40):
            s, rid = p.alloc_private(100)
            with lock:
                got.append(set(s.tolist()))
    ts = [threading.Thread(target=worker) for _ in range(8)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    allslots = [x for g in got for x in g]
    assert len(allslots) == len(set(allslots)) == 320 * 100
