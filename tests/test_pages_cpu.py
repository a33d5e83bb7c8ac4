"""The host page allocator of continuous batching (mk_pages_* in mk.h), on
the CPU: admission, growth page by page, retirement and reuse, the scratch
page of free rows, and the errors for bad states and an exhausted pool."""
import numpy as np

import persistent_decode_megakernel_04_b300 as mk


def test_admit_extend_retire_and_reuse():
    pool = mk.PagePool(num_pages=9, batch=3, max_pages=4, page_size=64)
    sp = pool.scratch_page
    assert sp == 8 and pool.free_count == 8
    assert np.all(pool.table() == sp)  # every row free: all entries name the scratch page
    assert pool.admit(0, 70) == mk.MK_OK  # 2 pages
    assert pool.admit(2, 1) == mk.MK_OK  # 1 page
    t = pool.table()
    assert sorted(t[0, :2].tolist() + t[2, :1].tolist()) == [0, 1, 2] and pool.free_count == 5
    assert np.all(t[0, 2:] == sp) and np.all(t[1] == sp) and np.all(t[2, 1:] == sp)
    assert pool.extend(0, 128) == mk.MK_OK and pool.free_count == 5  # still 2 pages
    assert pool.extend(0, 129) == mk.MK_OK and pool.free_count == 4  # a third page
    first = pool.table()[0, :3].tolist()
    assert len(set(first)) == 3 and sp not in first
    assert pool.retire(0) == mk.MK_OK and pool.free_count == 7
    assert np.all(pool.table()[0] == sp)
    assert pool.admit(1, 256) == mk.MK_OK and pool.free_count == 3  # reuses freed pages
    assert set(pool.table()[1].tolist()) <= set(range(8))
    pool.close()


def test_bad_states_and_exhaustion_are_errors_that_change_nothing():
    pool = mk.PagePool(num_pages=4, batch=2, max_pages=2, page_size=64)
    assert pool.extend(0, 10) == mk.MK_ERR_INVALID  # not admitted
    assert pool.retire(1) == mk.MK_ERR_INVALID
    assert pool.admit(0, 129) == mk.MK_ERR_INVALID  # 3 pages > max_pages
    assert pool.admit(5, 1) == mk.MK_ERR_INVALID and pool.admit(0, 0) == mk.MK_ERR_INVALID
    assert pool.admit(0, 100) == mk.MK_OK and pool.admit(0, 1) == mk.MK_ERR_INVALID  # already live
    assert pool.free_count == 1
    before = pool.table().copy()
    assert pool.admit(1, 100) == mk.MK_ERR_OOM  # needs 2, 1 free
    assert np.array_equal(pool.table(), before) and pool.free_count == 1
    assert pool.admit(1, 64) == mk.MK_OK and pool.free_count == 0
    assert pool.extend(1, 65) == mk.MK_ERR_OOM
    pool.close()
