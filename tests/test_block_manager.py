"""The host block manager (pa_bm_*) against the pages' worked example and a
plain-Python model of the same operations over random operation sequences."""
import json
import os
import random

import numpy as np
import pytest

from block_manager_ref import LATER, NEVER, OK, RefBlockManager
from paged_kv_cache_168_gb300 import _lib, build as build_mod
from paged_kv_cache_168_gb300._lib import BlockManager, PagedKVError

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_mod.build()


def test_cow_worked_example():
    ex = json.load(open(os.path.join(GOLDEN, "cow_worked_example.json")))
    bs = ex["block_size"]
    bm = BlockManager(bs, 6)
    prompt = list(range(ex["prompt_tokens"]))
    bm.allocate(0, prompt)                             # sequence A
    bm.fork(0, 1)                                      # B and C share A's prompt blocks
    bm.fork(0, 2)
    p0, p1 = bm.block_table(0)[0]
    assert bm.ref_count(p0) == 3 and bm.ref_count(p1) == 3
    names = {"A": 0, "B": 1, "C": 2}
    new_blocks = {}
    for name in ex["write_order"]:
        slot, cow = bm.append_slot(names[name], 1000 + names[name])
        expected = ex["expected_copy_pairs"][name]
        if expected:
            assert cow is not None and cow[0] == p1    # the shared prompt block is copied
            new_blocks[name] = cow[1]
            assert slot == cow[1] * bs + ex["expected_new_token_position"]["block_offset"]
        else:
            assert cow is None and slot == p1 * bs + ex["expected_new_token_position"]["block_offset"]
    # the example's final tables and counts, with its block ids relabelled
    relabel = {0: p0, 1: p1, 2: new_blocks["A"], 3: new_blocks["B"]}
    for name, table in ex["expected_tables"].items():
        assert bm.block_table(names[name])[0].tolist() == [relabel[b] for b in table]
    for b, count in ex["expected_ref_counts"].items():
        assert bm.ref_count(relabel[int(b)]) == count


def test_admission_statuses():
    bm = BlockManager(16, 10, watermark=0.1)           # 1 block kept free
    assert bm.can_allocate(16 * 10) == NEVER
    assert bm.can_allocate(16 * 9) == OK
    bm.allocate(0, list(range(16 * 5)))
    assert bm.can_allocate(16 * 5) == LATER
    assert bm.can_allocate(16 * 4) == OK
    with pytest.raises(PagedKVError) as e:
        bm.allocate(1, list(range(16 * 6)))
    assert e.value.status == _lib.PA_ERR_OUT_OF_BLOCKS and bm.num_free() == 5   # nothing changed


def test_sliding_window_tables_wrap():
    bm = BlockManager(16, 8, sliding_window=40)        # ceil(40/16) = 3 blocks
    bm.allocate(0, list(range(100)))                   # 7 logical blocks
    table, n = bm.block_table(0)
    assert n == 100 and len(table) == 7
    assert [table[i] for i in range(7)] == [table[i % 3] for i in range(7)]
    assert bm.num_free() == 5
    slot, cow = bm.append_slot(0, 7)
    assert cow is None and slot == table[100 // 16 % 3] * 16 + 100 % 16


def test_prefix_caching_shares_full_blocks_and_evicts_lru():
    bm = BlockManager(4, 6, prefix_caching=True)
    bm.allocate(0, [1, 2, 3, 4, 5, 6, 7, 8, 9])        # two full blocks + one partial
    bm.allocate(1, [1, 2, 3, 4, 5, 6, 7, 8, 10, 11])   # same first two blocks
    t0, t1 = bm.block_table(0)[0], bm.block_table(1)[0]
    assert t0[:2].tolist() == t1[:2].tolist() and t0[2] != t1[2]
    assert bm.ref_count(int(t0[0])) == 2
    bm.allocate(2, [1, 2, 3, 4, 9, 9, 9, 9])           # first block shared, second differs
    t2 = bm.block_table(2)[0]
    assert t2[0] == t0[0] and t2[1] != t0[1]
    bm.free(0)
    bm.free(1)
    bm.free(2)
    assert bm.num_free() == 6                          # cached blocks count as free
    bm.allocate(3, [1, 2, 3, 4, 5, 6, 7, 8])           # revived from the evictor
    assert bm.block_table(3)[0].tolist() == t0[:2].tolist()


@pytest.mark.parametrize("seed,caching,window", [(s, c, w) for s in range(6) for c, w in
                                                  ((False, 0), (True, 0), (False, 24))])
def test_random_operations_match_the_model(seed, caching, window):
    rnd = random.Random(seed)
    bs, ngpu, ncpu = 4, 40, 30
    cpp = BlockManager(bs, ngpu, ncpu, watermark=0.05, sliding_window=window, prefix_caching=caching)
    ref = RefBlockManager(bs, ngpu, ncpu, watermark=0.05, window=window, caching=caching)
    alive, swapped, next_id = [], [], 0
    vocab = [1, 2, 3] if caching else list(range(50))
    for step in range(300):
        op = rnd.random()
        if op < 0.25 or not alive:
            n = rnd.randint(1, 14)
            toks = [rnd.choice(vocab) for _ in range(n)]
            assert cpp.can_allocate(n) == ref.can_allocate(n)
            try:
                ref.allocate(next_id, toks)
            except MemoryError:
                with pytest.raises(PagedKVError):
                    cpp.allocate(next_id, toks)
                continue
            cpp.allocate(next_id, toks)
            alive.append(next_id)
            next_id += 1
        elif op < 0.6:
            sid = rnd.choice(alive)
            tok = rnd.choice(vocab)
            try:
                want = ref.append_slot(sid, tok)
            except MemoryError:
                continue            # the model ran dry mid-way; stop comparing this sequence
            got = cpp.append_slot(sid, tok)
            assert got == want, (step, sid)
        elif op < 0.7:
            sid = rnd.choice(alive)
            ref.fork(sid, next_id)
            cpp.fork(sid, next_id)
            alive.append(next_id)
            next_id += 1
        elif op < 0.85:
            sid = alive.pop(rnd.randrange(len(alive)))
            ref.free(sid)
            cpp.free(sid)
        elif op < 0.93 and alive and ncpu and not caching:
            sid = rnd.choice(alive)
            need = len(set(ref.block_table(sid)[0]))
            assert cpp.can_swap_out([sid]) == ref.can_swap_out([sid]) == (ref.cpu.num_free() >= need)
            if ref.cpu.num_free() >= need:
                assert cpp.swap_out([sid]).tolist() == [list(p) for p in ref.swap_out([sid])]
                alive.remove(sid)
                swapped.append(sid)
        elif swapped:
            sid = swapped.pop(0)
            need = len(set(ref.block_table(sid)[0]))
            assert cpp.can_swap_in([sid]) == ref.can_swap_in([sid])
            if ref.gpu.num_free() >= need:
                assert cpp.swap_in([sid]).tolist() == [list(p) for p in ref.swap_in([sid])]
                alive.append(sid)
            else:
                swapped.insert(0, sid)
        for sid in alive + swapped:
            t, n = cpp.block_table(sid)
            rt, rn = ref.block_table(sid)
            assert t.tolist() == rt and n == rn, (step, sid)
        assert cpp.num_free() == ref.gpu.num_free()
        assert [cpp.ref_count(b) for b in range(ngpu)] == ref.gpu.ref
        k = rnd.randint(0, len(alive) + 3)
        assert cpp.can_append_slots(k) == ref.can_append_slots(k)


def test_swap_and_append_admission():
    # two sequences share both blocks of a prompt (a fork): swapping them
    # together needs those two blocks once on the other side
    bm = BlockManager(4, 6, 2, watermark=0.0)
    bm.allocate(0, list(range(8)))                  # 2 full blocks
    bm.fork(0, 1)
    assert bm.can_swap_out([0, 1]) and bm.can_swap_out([0])
    bm.allocate(2, [1])                             # 1 block
    assert not bm.can_swap_out([0, 1, 2])           # 3 distinct blocks, 2 host blocks
    assert bm.can_append_slots(3) and bm.can_append_slots(bm.num_free())
    assert not bm.can_append_slots(bm.num_free() + 1)
    pairs = bm.swap_out([0, 1])
    assert len(pairs) == 2 and bm.num_free(on_host=True) == 0
    assert bm.can_swap_in([0, 1]) == OK    # 5 device blocks free, 2 needed
    bm.allocate(3, list(range(16)))                 # 4 blocks: 1 left
    assert bm.can_swap_in([0, 1]) == LATER
    bm.free(3)
    with pytest.raises(PagedKVError):
        bm.can_swap_in([2])                         # not swapped out
    with pytest.raises(PagedKVError):
        bm.can_swap_out([0])                        # swapped out
    with pytest.raises(PagedKVError):
        bm.can_swap_in([99])                        # unknown
    # the watermark keeps admission from taking the last free blocks; a request
    # larger than the pool less the watermark can never be admitted
    wm = BlockManager(4, 10, 10, watermark=0.2)     # 2 blocks held back
    wm.allocate(0, list(range(36)))                 # 9 blocks
    wm.swap_out([0])
    assert wm.can_swap_in([0]) == NEVER    # 10 - 9 < 2
    wm2 = BlockManager(4, 10, 10, watermark=0.2)
    wm2.allocate(0, list(range(32)))                # 8 blocks
    wm2.swap_out([0])
    assert wm2.can_swap_in([0]) == OK      # 10 free - 8 >= 2
    wm2.allocate(1, [5])
    assert wm2.can_swap_in([0]) == LATER   # 9 free - 8 < 2


def test_errors_leave_state_unchanged():
    bm = BlockManager(8, 4)
    with pytest.raises(PagedKVError):
        bm.append_slot(7, 1)                           # unknown sequence
    bm.allocate(0, [1, 2, 3])
    with pytest.raises(PagedKVError):
        bm.allocate(0, [1])                            # id in use
    with pytest.raises(PagedKVError):
        bm.fork(0, 0)
    with pytest.raises(PagedKVError):
        BlockManager(8, 4, sliding_window=16, prefix_caching=True)
    assert bm.block_table(0)[0].size == 1
