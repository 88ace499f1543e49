"""Host block manager: free list, reserve on admit, prefix sharing, COW.

Pinned by the block arithmetic the pages state (tests/golden/page_arithmetic.json)
and by invariants (no block is both free and referenced; nothing is partially
allocated on failure; blocks return at reference count zero).
"""
import json
import os

import numpy as np
import pytest

from paged_kv_cache_06_gb300.block_manager import BlockManager
from paged_kv_cache_06_gb300.ops import PagedKVError

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_arithmetic.json")))

NO_BLOCKS, NOT_FOUND, STATE = 6, 7, 8


def _invariants(bm: BlockManager, seqs):
    st = bm.stats()
    refs = np.array([bm.refcount(b) for b in range(bm.num_blocks)])
    assert st["free_blocks"] == int((refs == 0).sum())
    assert st["used_blocks"] == bm.num_blocks - st["free_blocks"]
    assert st["shared_blocks"] == int((refs > 1).sum())
    for s in seqs:
        row, n = bm.table(s)
        used = row[row >= 0]
        assert np.all(refs[used] >= 1)


def test_largest_request_needs_68_blocks():
    g = G["largest_request"]
    bm = BlockManager(1000, g["block_size"], 128)
    bm.admit(1, g["prompt"], g["budget"], reserve=True)
    assert bm.stats()["used_blocks"] == g["blocks"]


def test_small_pool_holds_292_blocks_and_four_largest_requests():
    g = G["small_pool"]
    per_token = g["layers"] * g["kv_heads"] * g["head_dim"] * g["elem_bytes"] * 2
    assert per_token == g["bytes_per_token"]
    nblocks = g["pool_bytes"] // (per_token * g["block_size"])
    assert nblocks == g["blocks"]
    bm = BlockManager(nblocks, g["block_size"], 128)
    admitted = [bm.try_admit(i, 4096, 256) for i in range(5)]
    # 4 x 68 = 272 <= 292 < 5 x 68: the fifth waits even though rows are free
    assert admitted == [True, True, True, True, False]
    assert bm.stats()["free_blocks"] == 292 - 4 * 68


def test_mean_rounding_waste_is_about_half_a_block():
    g = G["rounding_waste"]
    bs = g["block_size"]
    bm = BlockManager(100000, bs, 1024)
    n = 0
    for need in range(1, 8 * bs + 1):  # every remainder equally often
        bm.admit(need, need, 0, reserve=True)
        n += 1
    waste = bm.stats()["reserved_slots"] / n
    assert abs(waste - (bs - 1) / 2) < 1e-9  # 31.5 tokens ~ "32 tokens"
    mb = waste * G["small_pool"]["bytes_per_token"] / 1e6
    assert round(mb, 1) == g["mean_waste_mb"]


@pytest.mark.parametrize("bs", [16, 256])
def test_shared_prompt_shares_whole_blocks_only(bs):
    g = G["shared_prompt"]
    bm = BlockManager(1000, bs, 1000)
    pid, ids = bm.register_prefix(g["prompt_tokens"])
    assert len(ids) * bs == g["shared_tokens"][str(bs)]


def test_internal_fragmentation_bounded_by_one_partial_block():
    g = G["fragmentation_bound"]
    bm = BlockManager(4096, g["block_size"], 512)
    for s, L in enumerate(range(1, 200)):
        bm.admit(s, L, 0, reserve=False)
        row, n = bm.table(s)
        empty = int((row >= 0).sum()) * g["block_size"] - n
        assert 0 <= empty <= g["max_empty_slots"]


def test_dense_table_size():
    g = G["dense_table"]
    assert g["context"] // g["block_size"] == g["entries_per_row"]
    bm = BlockManager(8, g["block_size"], g["entries_per_row"])
    bm.admit(0, 5, 0)
    t, lens = bm.tables([0] * g["rows"])
    assert t.nbytes == g["bytes"] and t.dtype == np.int32


def test_request_a_blocks_and_shared_preamble():
    g = G["request_a"]
    bs = g["block_size"]
    bm = BlockManager(200, bs, 64)
    pid, ids = bm.register_prefix(g["prefix_tokens"])
    assert len(ids) == g["shared_blocks"]
    bm.admit(1, g["tokens"], 0, prefix_id=pid)
    row, n = bm.table(1)
    assert int((row >= 0).sum()) == g["blocks"] and n == g["tokens"]
    assert np.array_equal(row[:g["shared_blocks"]], ids)
    bm.admit(2, g["tokens"], 0, prefix_id=pid)
    row2, _ = bm.table(2)
    assert np.array_equal(row2[:g["shared_blocks"]], ids)
    assert set(row2[g["shared_blocks"]:40]).isdisjoint(set(row[g["shared_blocks"]:40]))
    assert bm.stats()["shared_blocks"] == g["shared_blocks"]


def test_free_list_is_lifo_and_eviction_only_edits_it():
    bm = BlockManager(8, 4, 8)
    bm.admit(0, 8, 0)          # takes 2 blocks
    row0, _ = bm.table(0)
    bm.free(0)
    bm.admit(1, 8, 0)          # gets the same blocks back (LIFO), no copy
    row1, _ = bm.table(1)
    assert set(row0[:2]) == set(row1[:2])
    assert bm.stats()["free_blocks"] == 6


def test_reserve_on_admit_is_all_or_nothing():
    bm = BlockManager(10, 4, 16)
    bm.admit(0, 16, 8)                     # 6 blocks
    before = bm.stats()
    with pytest.raises(PagedKVError) as e:
        bm.admit(1, 8, 12)                 # needs 5 > 4 free
    assert e.value.status == NO_BLOCKS
    assert bm.stats() == before            # nothing partially allocated
    bm.admit(1, 8, 8)                      # 4 blocks fit exactly
    assert bm.stats()["free_blocks"] == 0
    # a reserved sequence never needs a block mid generation
    for _ in range(8):
        bm.append_slot(0)
        bm.append_slot(1)
    with pytest.raises(PagedKVError) as e:
        bm.append_slot(1)                  # budget spent, pool empty
    assert e.value.status == NO_BLOCKS


def test_growth_one_block_at_a_time_without_reservation():
    bm = BlockManager(4, 4, 8)
    bm.admit(0, 3, 100, reserve=False)     # one block, nothing reserved
    assert bm.stats()["used_blocks"] == 1
    positions = [bm.append_slot(0)[0] for _ in range(9)]
    assert positions == list(range(3, 12))
    assert bm.stats()["used_blocks"] == 3  # 12 tokens -> 3 blocks of 4
    row, n = bm.table(0)
    assert n == 12 and int((row >= 0).sum()) == 3


def test_prefix_refcount_and_copy_on_write():
    bm = BlockManager(64, 16, 64)
    pid, ids = bm.register_prefix(600)                 # 600 // 16 = 37 whole blocks
    assert len(ids) == 37
    bm.admit(10, 100, 4, prefix_id=pid)                 # prompt ends inside shared block 6
    bm.admit(11, 100, 0, prefix_id=pid)
    assert bm.refcount(int(ids[6])) == 3               # registration + two sequences
    pos, cow = bm.append_slot(10)
    assert pos == 100 and cow is not None and cow[0] == ids[6]
    row, n = bm.table(10)
    assert row[6] == cow[1] and row[6] != ids[6] and n == 101
    assert bm.refcount(int(ids[6])) == 2
    pos, cow2 = bm.append_slot(10)                     # now private: no second copy
    assert cow2 is None
    assert bm.stats()["cow_copies"] == 1
    _invariants(bm, [10, 11])
    bm.release_prefix(pid)
    bm.free(11)
    # blocks 0..5 still referenced by seq 10; block ids[6] and 7.. freed
    assert bm.refcount(int(ids[0])) == 1 and bm.refcount(int(ids[6])) == 0
    bm.free(10)
    assert bm.stats()["free_blocks"] == 64
    _invariants(bm, [])


def test_sole_owner_of_a_prefix_block_writes_in_place():
    bm = BlockManager(16, 4, 8)
    pid, ids = bm.register_prefix(8)
    bm.admit(0, 6, 2, prefix_id=pid, reserve=True)
    bm.release_prefix(pid)                              # seq 0 is now the only owner
    pos, cow = bm.append_slot(0)
    assert pos == 6 and cow is None


def test_fault_injection_pop_failure_reports_no_blocks():
    bm = BlockManager(32, 4, 16)
    bm.inject_pop_failure(3)
    with pytest.raises(PagedKVError) as e:
        bm.admit(0, 16, 0)                              # needs 4 pops, 3 allowed
    assert e.value.status == NO_BLOCKS
    assert bm.stats()["used_blocks"] == 0
    bm.admit(0, 12, 0)                                  # 3 pops fine
    with pytest.raises(PagedKVError):
        bm.append_slot(0)                               # position 12 needs a 4th block
    assert bm.table(0)[1] == 12                         # length unchanged
    bm.inject_pop_failure(-1)
    assert bm.append_slot(0)[0] == 12


def test_errors_for_unknown_ids_and_states():
    bm = BlockManager(8, 4, 2)
    with pytest.raises(PagedKVError) as e:
        bm.free(99)
    assert e.value.status == NOT_FOUND
    with pytest.raises(PagedKVError) as e:
        bm.release_prefix(3)
    assert e.value.status == NOT_FOUND
    bm.admit(0, 7, 1)
    with pytest.raises(PagedKVError) as e:
        bm.admit(0, 1, 0)
    assert e.value.status == STATE
    bm.append_slot(0)
    with pytest.raises(PagedKVError) as e:
        bm.append_slot(0)                               # past max_blocks_per_row * bs
    assert e.value.status in (STATE, NO_BLOCKS)
    with pytest.raises(PagedKVError):
        bm.admit(1, 9, 0)                               # cannot fit its table
