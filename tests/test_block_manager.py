"""Host block manager: the page-1 demo's end state, invariants and failure paths."""
import math
import random

import numpy as np
import pytest

from conftest import read_golden
from paged_kv_cache_170_gb300.block_manager import BlockManager, BlockManagerError, PoolExhausted
from paged_kv_cache_170_gb300 import scenarios
from paged_kv_cache_170_gb300.workloads import LONGCTX, PREFIX, scaled


def _run_demo():
    """The operation sequence of aiqz.cc's "Python 演示" section."""
    mgr = BlockManager(12, 4)
    cows = []
    mgr.allocate("sys", 8)
    mgr.fork("A", "sys", 8)
    for _ in range(3):
        cows.append(mgr.append_slot("A")[1])
    mgr.fork("B", "sys", 8)
    for _ in range(2):
        cows.append(mgr.append_slot("B")[1])
    mgr.fork("C", "A", 9)
    slot, cow = mgr.append_slot("C")
    cows.append(cow)
    return mgr, cows, slot


def test_demo_end_state_matches_golden():
    mgr, cows, slot = _run_demo()
    g = {}
    for row in read_golden("demo_block_manager.txt"):
        g.setdefault(row[0], []).append(row[1:])
    assert mgr.refs == [int(x) for x in g["refs"][0]]
    for name, *ids in g["table"]:
        assert mgr.tables[name] == [int(x) for x in ids]
    for name, n in g["used"]:
        assert mgr.used[name] == int(n)
    no_share = sum(math.ceil(mgr.used[r] / mgr.block_size) for r in mgr.tables)
    assert no_share == int(g["no_share"][0][0])
    assert mgr.num_used_blocks() == int(g["paged_shared"][0][0])
    # only C's write copied: A's third block (2) into the fresh block 4,
    # and C's token 9 lands at offset 1 of block 4
    assert [c for c in cows if c is not None] == [(2, 4)]
    assert slot == 4 * 4 + 1
    mgr.check()


def test_fresh_block_when_last_is_full_never_copies():
    mgr = BlockManager(8, 4)
    mgr.allocate("a", 4)
    mgr.fork("b", "a")
    slot, cow = mgr.append_slot("b")       # last block full and shared: new block, no copy
    assert cow is None and mgr.tables["b"] == [0, 1] and slot == 4
    assert mgr.refs[:2] == [2, 1]


def test_cow_then_exclusive_writes_in_place():
    mgr = BlockManager(8, 4)
    mgr.allocate("a", 6)
    mgr.fork("b", "a")
    _, cow = mgr.append_slot("a")         # shared tail: copy
    assert cow == (1, 2) and mgr.refs[1] == 1 and mgr.refs[2] == 1
    _, cow = mgr.append_slot("b")         # tail now exclusive: in place
    assert cow is None and mgr.tables["b"] == [0, 1]
    mgr.check()


def test_free_returns_blocks_only_at_zero():
    mgr = BlockManager(6, 2)
    mgr.allocate("a", 4)
    mgr.fork("b", "a")
    mgr.free_seq("a")
    assert mgr.num_free() == 4 and mgr.refs[:2] == [1, 1]
    mgr.free_seq("b")
    assert mgr.num_free() == 6 and list(mgr.free)[-2:] == [0, 1]
    mgr.check()
    with pytest.raises(BlockManagerError):
        mgr.free_seq("b")   # double free


def test_exhaustion_leaves_state_unchanged():
    mgr = BlockManager(3, 4)
    mgr.allocate("a", 8)
    mgr.fork("b", "a", 6)
    before = (list(mgr.refs), {k: list(v) for k, v in mgr.tables.items()}, dict(mgr.used), list(mgr.free))
    with pytest.raises(PoolExhausted):
        mgr.allocate("c", 9)
    mgr.append_slot("b")  # copies block 1 into block 2 (the last free one)
    mgr.fork("d", "b")
    snapshot = (list(mgr.refs), {k: list(v) for k, v in mgr.tables.items()}, dict(mgr.used), list(mgr.free))
    with pytest.raises(PoolExhausted):
        mgr.append_slot("d")  # needs a copy, pool empty
    assert snapshot == (list(mgr.refs), {k: list(v) for k, v in mgr.tables.items()}, dict(mgr.used),
                        list(mgr.free))
    assert before != snapshot
    mgr.check()


def test_random_operations_keep_audit_consistent():
    rng = random.Random(0)
    mgr = BlockManager(64, 4, free_order=rng.sample(range(64), 64))
    live = []
    for step in range(3000):
        op = rng.random()
        try:
            if op < 0.15 or not live:
                name = ("s", step)
                mgr.allocate(name, rng.randint(0, 12))
                live.append(name)
            elif op < 0.3:
                parent = rng.choice(live)
                name = ("f", step)
                mgr.fork(name, parent, rng.randint(0, mgr.used[parent]))
                live.append(name)
            elif op < 0.85:
                mgr.append_slot(rng.choice(live))
            else:
                victim = rng.choice(live)
                mgr.free_seq(victim)
                live.remove(victim)
        except PoolExhausted:
            victim = rng.choice(live)
            mgr.free_seq(victim)
            live.remove(victim)
        mgr.check()
    # slots handed out by append are always inside the sequence's own last block
    s = live[0]
    slot, _ = mgr.append_slot(s)
    assert slot // 4 == mgr.tables[s][-1]


def test_shared_prefix_scenario_structure():
    inp = scenarios.shared_prefix_inputs(seed=0, num_parents=6, prefix_tokens=64, suffix_max=100,
                                         w=scaled(PREFIX, num_blocks=128, max_blocks_per_seq=16))
    mgr = inp.extra["manager"]
    mgr.check()
    pairs = inp.copy_pairs.numpy()
    # the first of each pair copied its shared tail, the second wrote in place
    assert pairs.shape == (6, 2)
    tables = inp.block_tables.numpy()
    lens = inp.context_lens.numpy()
    assert np.all(lens[0::2] == lens[1::2])
    prefix_blocks = tables[0, :4]
    assert np.all(tables[:, :4] == prefix_blocks)
    assert all(mgr.refs[p] == 12 for p in prefix_blocks)
    for i in range(6):
        n = -(-int(lens[2 * i]) // 16)
        a, b = tables[2 * i, :n], tables[2 * i + 1, :n]
        assert a[-1] != b[-1] and a[-1] == pairs[i, 1] and b[-1] == pairs[i, 0]
    assert np.array_equal(inp.extra["manager_slots"].numpy() // 16,
                          tables[np.arange(12), (lens - 1) // 16])


def test_long_context_scenario_structure():
    inp = scenarios.long_context_inputs(seed=0, num_prompts=2, branches=3, prompt_tokens=96, suffix_max=40,
                                        w=scaled(LONGCTX, num_blocks=64, max_blocks_per_seq=8))
    mgr = inp.extra["manager"]
    mgr.check()
    assert inp.copy_pairs.shape[0] == 0          # branches start at a block boundary
    tables = inp.block_tables.numpy()
    assert np.all(tables[0:3, :3] == tables[0, :3]) and np.all(tables[3:6, :3] == tables[3, :3])
    assert all(mgr.refs[p] == 3 for p in tables[0, :3])
