"""The pages' memory figures (pool_report) and the contiguous allocation
policy of the block manager (host only, no GPU)."""
import numpy as np
import pytest

from paged_kv_cache_170_gb300 import scenarios
from paged_kv_cache_170_gb300.block_manager import BlockManager, pool_report


def test_report_on_a_hand_checked_fork():
    # B = 4: A holds 8 tokens (2 full blocks); B forks all of them; A grows
    # by 2 tokens, B by 3 (each into a block of its own).
    mgr = BlockManager(16, 4)
    mgr.allocate("A", 8)
    mgr.fork("B", "A")
    for _ in range(2):
        mgr.append_slot("A")
    for _ in range(3):
        mgr.append_slot("B")
    tables = mgr.block_tables(["A", "B"])
    lens = mgr.context_lens(["A", "B"])
    bpt = 10  # bytes per token
    r = pool_report(tables, lens, 4, bpt, max_len=16)
    assert r["blocks_distinct"] == 4 and r["blocks_referenced"] == 6
    assert r["m_alloc_bytes"] == 4 * 4 * bpt
    assert r["m_used_bytes"] == (4 + 4 + 2 + 3) * bpt
    assert r["eta_waste"] == pytest.approx(3 / 16)
    # the pages' formula: N_p = 2 shared blocks, R = 2 sharers
    assert r["m_saved_bytes"] == 2 * 4 * bpt * (2 - 1)
    assert r["eta_prime_estimate"] == pytest.approx((1 / 6 + 1 / 6) / 2)
    assert r["contiguous_reserved_bytes"] == 2 * 16 * bpt
    assert r["contiguous_utilisation"] == pytest.approx(21 / 32)


def test_saved_memory_matches_the_pages_formula_for_one_shared_prefix():
    # R requests forked from one parent holding N_p full blocks, each then
    # writing into a block of its own: M_saved = N_p * B * bytes * (R - 1)
    B, Np, R, bpt = 16, 5, 7, 4096
    mgr = BlockManager(200, B)
    mgr.allocate(0, Np * B)
    for r in range(1, R):
        mgr.fork(r, 0)
    for r in range(R):
        for _ in range(r + 1):
            mgr.append_slot(r)
    seqs = list(range(R))
    rep = pool_report(mgr.block_tables(seqs), mgr.context_lens(seqs), B, bpt)
    assert rep["m_saved_bytes"] == Np * B * bpt * (R - 1)


def test_waste_of_paged_allocation_follows_the_half_block_estimate():
    # N blocks per request, the last one filled uniformly: waste ~ half a block
    rng = np.random.default_rng(0)
    B, N, S = 16, 8, 4000
    lens = (N - 1) * B + rng.integers(1, B + 1, size=S)
    tables = np.arange(S * N).reshape(S, N)
    rep = pool_report(tables, lens, B, 1)
    assert rep["eta_prime_estimate"] == pytest.approx(1 / (2 * N))
    # exact expectation of the waste ratio: (B - 1) / 2 empty slots of N * B
    assert rep["eta_waste"] == pytest.approx((B - 1) / (2 * N * B), rel=0.05)


def test_shared_prefix_workload_report():
    inp = scenarios.shared_prefix_inputs(0)
    bpt = 2 * 8 * 128 * 2
    rep = pool_report(inp.block_tables.numpy(), inp.context_lens.numpy(), 16, bpt, max_len=2048)
    # the 1024-token prefix is shared by all 128 requests: at least the pages' saving
    assert rep["m_saved_bytes"] >= 64 * 16 * bpt * (128 - 1)
    assert 0.0 <= rep["eta_waste"] < 0.1 and rep["paged_utilisation"] > 0.9


def test_contiguous_policy_keeps_sequences_together():
    mgr = BlockManager(64, 4, policy="contiguous")
    a = mgr.allocate("a", 10)  # 3 blocks
    b = mgr.allocate("b", 16)  # 4 blocks
    assert a == [0, 1, 2] and b == [3, 4, 5, 6]
    for _ in range(3):  # a's last block has 2 free slots, then a new block: 3 is taken, so the lowest free
        mgr.append_slot("a")
    assert mgr.tables["a"] == [0, 1, 2, 7]
    mgr.free_seq("b")
    c = mgr.allocate("c", 12)  # first run of 3 free ids
    assert c == [3, 4, 5]
    for _ in range(4 * 3):
        mgr.append_slot("c")  # grows into 6, then 8, 9 (7 is a's)
    assert mgr.tables["c"] == [3, 4, 5, 6, 8, 9]
    mgr.check()


@pytest.mark.parametrize("policy", ["queue", "contiguous"])
def test_random_operations_keep_the_manager_consistent(policy):
    rng = np.random.default_rng(7)
    mgr = BlockManager(300, 8, free_order=rng.permutation(300).tolist(), policy=policy)
    live, next_id = [], 0
    for _ in range(2000):
        op = rng.integers(0, 4)
        try:
            if op == 0 or not live:
                mgr.allocate(next_id, int(rng.integers(1, 60)))
                live.append(next_id)
                next_id += 1
            elif op == 1:
                parent = live[int(rng.integers(len(live)))]
                mgr.fork(next_id, parent)
                live.append(next_id)
                next_id += 1
            elif op == 2:
                mgr.append_slot(live[int(rng.integers(len(live)))])
            else:
                mgr.free_seq(live.pop(int(rng.integers(len(live)))))
        except Exception as e:  # a full pool leaves the state unchanged
            assert type(e).__name__ == "PoolExhausted"
        mgr.check()
