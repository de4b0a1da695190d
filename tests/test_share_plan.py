"""The shared-block decode plan (pa_share_plan, host code: no GPU needed).

Structural checks of the plan against the block tables it was built from,
and a float64 numpy walk through the plan -- partial states per piece and
row (shared groups, and each sequence's own group of private blocks), then
the merge -- that must reproduce the oracle's decode: the plan's split of the
work is complete and does not overlap.  (The GPU tests then check the
kernels that follow the plan.)
"""
import math

import numpy as np
import pytest
import torch

from oracle import reference
from paged_kv_cache_170_gb300 import build, scenarios
from paged_kv_cache_170_gb300 import workloads as W
from paged_kv_cache_170_gb300.block_manager import BlockManager

PASS_ROWS = 32  # query rows of a shared group's pass
OWN_PASS_ROWS = 8  # of an own group's pass
TC_MIN_ROWS = 32  # query rows per kv head from which a shared group goes to the tensor-core kernel
TC_ITEM_ROWS = 128  # rows of one of its work items


@pytest.fixture(scope="module")
def ops():
    build.build()
    from paged_kv_cache_170_gb300 import ops as _ops

    return _ops


def _prefix_small(seed=0):
    return scenarios.shared_prefix_inputs(seed, num_parents=4, prefix_tokens=256, suffix_max=300,
                                          w=W.scaled(W.PREFIX, num_blocks=300, max_blocks_per_seq=40))


def _longctx_small(seed=0):
    return scenarios.long_context_inputs(seed, num_prompts=2, branches=3, prompt_tokens=2048, suffix_max=200,
                                         w=W.scaled(W.LONGCTX, num_blocks=200, max_blocks_per_seq=80))


def _beam_like(seed=0):
    """A deeper trie: one root prompt, forked twice, each child forked again,
    with appends between forks (groups nest three levels)."""
    B, Hkv, Hq, D, NB = 16, 2, 8, 64, 400
    g = torch.Generator().manual_seed(seed)
    mgr = BlockManager(NB, B, free_order=torch.randperm(NB, generator=g).tolist())
    mgr.allocate(0, 16 * 6)  # 6 full blocks
    for child, parent in [(1, 0), (2, 0)]:
        mgr.fork(child, parent)
    for s in (0, 1, 2):
        for _ in range(16 * (s + 1) + 3):
            mgr.append_slot(s)
    for child, parent in [(3, 1), (4, 2), (5, 2)]:
        mgr.fork(child, parent)
    for s in range(6):
        for _ in range(5 + 7 * s):
            mgr.append_slot(s)
    S = 6
    tables = torch.as_tensor(mgr.block_tables(list(range(S)), 40, pad=0), dtype=torch.int32)
    lens = torch.as_tensor(mgr.context_lens(list(range(S))), dtype=torch.int32)
    q = torch.randn(S, Hq, D, generator=g).to(torch.bfloat16)
    kc = torch.randn(NB, Hkv, B, D, generator=g).to(torch.bfloat16)
    vc = torch.randn(NB, Hkv, B, D, generator=g).to(torch.bfloat16)
    return q, kc, vc, tables, lens, 1.0 / math.sqrt(D)


def _case(name):
    if name == "beam":
        return _beam_like()
    if name == "longctx4":  # four branches x 8 heads = 32 rows per kv head: the tensor cores take the prompts
        inp = scenarios.long_context_inputs(0, num_prompts=2, branches=4, prompt_tokens=2048, suffix_max=200,
                                            w=W.scaled(W.LONGCTX, num_blocks=220, max_blocks_per_seq=80))
        return inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale
    inp = _prefix_small() if name == "prefix" else _longctx_small()
    # the plan is built from the tables as the decode sees them (after the step's copies / writes)
    return inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale


def _check_structure(f, tables, lens, B, Hq, Hkv):
    S = tables.shape[0]
    Gq = Hq // Hkv
    full = [int(L) // B for L in lens]
    nb = [-(-int(L) // B) for L in lens]
    moff, mem = f["g_moff_arr"], f["g_members_arr"]
    b0, b1 = f["g_b0_arr"], f["g_b1_arr"]
    start = f["s_start_arr"]
    nsg = f["num_shared_groups"]
    own_of = {}
    for g in range(f["num_groups"]):
        members = mem[moff[g]:moff[g + 1]]
        assert 0 <= b0[g] < b1[g]
        if g >= nsg:  # own group: one sequence's private blocks, to its last (partial) block
            assert len(members) == 1 and members[0] not in own_of
            s = members[0]
            own_of[s] = g
            assert (b0[g], b1[g]) == (start[s], nb[s])
            assert f["g_prows_arr"][g] == OWN_PASS_ROWS
            assert f["g_passes_arr"][g] == -(-Gq // OWN_PASS_ROWS)
            continue
        assert len(members) >= 2 and list(members) == sorted(set(members))
        for s in members:
            assert full[s] >= b1[g], "a group block must be full for every member"
            assert np.array_equal(tables[s, b0[g]:b1[g]], tables[members[0], b0[g]:b1[g]])
        # maximal: the run cannot be extended by one block
        e = b1[g]
        extendable = all(full[s] > e for s in members) and len({int(tables[s, e]) for s in members}) == 1
        assert not extendable, f"group {g} could extend past block {e}"
        assert f["g_prows_arr"][g] == PASS_ROWS
        assert f["g_passes_arr"][g] == -(-len(members) * Gq // PASS_ROWS)
    # every sequence with tokens past its shared blocks has its own group
    assert set(own_of) == {s for s in range(S) if nb[s] > start[s]}
    assert f["own_tiles"] == int(bool(own_of))
    # memberships of each sequence chain from block 0 to its last block
    for s in range(S):
        ks = range(f["s_moff_arr"][s], f["s_moff_arr"][s + 1])
        runs = sorted((b0[f["s_mgroup_arr"][k]], b1[f["s_mgroup_arr"][k]]) for k in ks)
        at = 0
        for x, y in runs:
            assert x == at
            at = y
        assert at == nb[s] and start[s] <= full[s] <= nb[s]
        for k in ks:  # member index points back at s
            g, i = f["s_mgroup_arr"][k], f["s_midx_arr"][k]
            assert mem[moff[g] + i] == s
    # trie property: two sequences with identical full blocks [0, k) share groups covering [0, k)
    for s1 in range(S):
        for s2 in range(s1 + 1, S):
            k = 0
            while k < min(full[s1], full[s2]) and tables[s1, k] == tables[s2, k]:
                k += 1
            g1 = {f["s_mgroup_arr"][j] for j in range(f["s_moff_arr"][s1], f["s_moff_arr"][s1 + 1])}
            g2 = {f["s_mgroup_arr"][j] for j in range(f["s_moff_arr"][s2], f["s_moff_arr"][s2 + 1])}
            covered = sum(b1[g] - b0[g] for g in g1 & g2)
            assert covered == k, (s1, s2, covered, k)
    # shared groups on the tensor cores (many sharers, whole-block steps)
    # follow the other shared groups
    G = f["num_groups"]
    is_tc = [g < nsg and B in (16, 32, 64) and (moff[g + 1] - moff[g]) * Gq >= TC_MIN_ROWS for g in range(G)]
    assert is_tc[:nsg] == sorted(is_tc[:nsg])
    # pieces: each unit's tiles exactly once, in order; CTA ranges balanced
    U, P, N = f["num_units"], f["num_pieces"], f["nctas"]
    poff = f["u_poff_arr"]
    for u in range(U):
        g = f["u_group_arr"][u]
        ps = range(poff[u], poff[u + 1])
        assert all(f["p_unit_arr"][p] == u for p in ps)
        t = 0
        for p in ps:
            assert f["p_t0_arr"][p] == t and f["p_t1_arr"][p] > t
            t = f["p_t1_arr"][p]
        assert t == b1[g] - b0[g]
        assert u == f["g_ubase_arr"][g] + f["u_kvh_arr"][u] * f["g_passes_arr"][g] + f["u_pass_arr"][u]
    # CTA ranges, one set per cost line (shared units, then own units):
    # contiguous, covering every tile of the line, balanced in cost (a tile of
    # a unit whose pass has <= 8, <= 16 or more rows costs 3, 4 or 5, and a
    # unit UNIT_COST once), to within one tile and one unit start
    UNIT_COST = 8
    TC_FIXED_COST, TC_STEP_COST = 36, 8  # a tensor-core item's time in step cost units: fixed + per step

    def cost(u):
        g = f["u_group_arr"][u]
        pr = f["g_prows_arr"][g]
        rows = min(pr, (moff[g + 1] - moff[g]) * Gq - f["u_pass_arr"][u] * pr)
        return 3 if rows <= 8 else (4 if rows <= 16 else 5)

    shared_units = [u for u in range(U) if f["u_group_arr"][u] < nsg and not is_tc[f["u_group_arr"][u]]]
    tc_units = [u for u in range(U) if is_tc[f["u_group_arr"][u]]]
    own_units = [u for u in range(U) if f["u_group_arr"][u] >= nsg]
    assert shared_units + tc_units + own_units == list(range(U))  # in this order
    # the tensor-core pieces lie between the two CTA lines
    tc_pieces = list(range(f["c_poff_arr"][N], f["c_opoff_arr"][0]))
    assert f["c_poff_arr"][0] == 0 and f["c_opoff_arr"][N] == P
    assert sorted(tc_pieces) == [p for u in tc_units for p in range(poff[u], poff[u + 1])]
    # The step's CTAs that start only once the tensor-core items are done
    # (the last n of them, n = items <= N) get an item's time C less of each
    # line: shares (W + n C) / N and that minus C, W the cost of both lines
    line_total = {id(units): sum((b1[f["u_group_arr"][u]] - b0[f["u_group_arr"][u]]) * cost(u) + UNIT_COST
                                 for u in units) for units in (shared_units, own_units)}
    W = sum(line_total.values())
    n = f["num_tc_items"]
    weights = [1] * N
    if 0 < n < N and W > 0:
        C = TC_FIXED_COST + f["tc_chunk_steps"] * TC_STEP_COST
        se, sl = W + n * C, W + n * C - C * N
        if sl < 0:
            se, sl = W * N // max(1, N - n), 0
        weights = [se] * (N - n) + [sl] * n
    cum = np.concatenate([[0], np.cumsum(weights)])
    for units, coff in ((shared_units, f["c_poff_arr"]), (own_units, f["c_opoff_arr"])):
        per_cta = [sum((f["p_t1_arr"][p] - f["p_t0_arr"][p]) * cost(f["p_unit_arr"][p]) +
                       (UNIT_COST if f["p_t0_arr"][p] == 0 else 0)
                       for p in range(coff[c], coff[c + 1])) for c in range(N)]
        total = line_total[id(units)]
        assert sum(per_cta) == total
        assert all(f["p_unit_arr"][p] in units for p in range(coff[0], coff[N]))
        if units:
            slack = UNIT_COST + max(cost(u) for u in units)
            done = np.cumsum(per_cta)
            for c in range(N):  # each CTA's range ends within a tile and a unit start of its weighted share
                assert abs(done[c] - total * cum[c + 1] / cum[N]) <= slack
    # a tensor-core group's units are all cut into the same chunks; every
    # tensor-core piece belongs to exactly one item, which names the pieces of
    # the passes of its 128 rows against one chunk
    for g in range(G):
        if not is_tc[g]:
            continue
        us = [u for u in tc_units if f["u_group_arr"][u] == g]
        cuts = {tuple((f["p_t0_arr"][p], f["p_t1_arr"][p]) for p in range(poff[u], poff[u + 1])) for u in us}
        assert len(cuts) == 1
    items = f["t_items_arr"].reshape(-1, 12)
    assert len(items) == f["num_tc_items"] and f["t_items"] % 4 == 0
    seen = []
    for it in items:
        g, kvh, row0, rows, leader, mo, blk0, ntile = (int(x) for x in it[:8])
        assert is_tc[g] and row0 % TC_ITEM_ROWS == 0 and 0 <= row0 < rows == (moff[g + 1] - moff[g]) * Gq
        assert leader == mem[moff[g]] and mo == moff[g] and ntile > 0
        for k in range(4):
            pas = row0 // PASS_ROWS + k
            p = int(it[8 + k])
            if pas >= f["g_passes_arr"][g]:
                assert p == -1
                continue
            u = f["g_ubase_arr"][g] + kvh * f["g_passes_arr"][g] + pas
            assert f["p_unit_arr"][p] == u
            assert (b0[g] + f["p_t0_arr"][p], f["p_t1_arr"][p] - f["p_t0_arr"][p]) == (blk0, ntile)
            seen.append(p)
    assert sorted(seen) == tc_pieces
    assert list(items[:, 7]) == sorted(items[:, 7], reverse=True)  # the longest chunks first
    # each item's q rows (sequence * Hq + head, -1 past the group's rows) and
    # physical blocks (-1 past its chunk), at fixed strides
    stride = f["t_blk_stride"]
    qrows = f["t_qrow_arr"].reshape(-1, TC_ITEM_ROWS)
    blks = f["t_blk_arr"].reshape(-1, stride) if stride else f["t_blk_arr"].reshape(0, 0)
    assert len(qrows) == len(items) and len(blks) == len(items)
    assert not len(items) or stride == f["tc_chunk_steps"] * (64 // B)
    for it, qr, bl in zip(items, qrows, blks):
        g, kvh, row0, rows, leader, mo, blk0, ntile = (int(x) for x in it[:8])
        want = [int(mem[moff[g] + r // Gq]) * Hq + kvh * Gq + r % Gq if r < rows else -1
                for r in range(row0, row0 + TC_ITEM_ROWS)]
        assert list(qr) == want
        assert list(bl) == [int(tables[leader, blk0 + j]) if j < ntile else -1 for j in range(stride)]
    # the packed descriptors repeat the piece's unit, tiles and group fields
    desc = f["p_desc_arr"].reshape(P, 12)
    for p in range(P):
        u = f["p_unit_arr"][p]
        g = f["u_group_arr"][u]
        assert list(desc[p]) == [u, f["p_t0_arr"][p], f["p_t1_arr"][p], g, f["u_kvh_arr"][u], f["u_pass_arr"][u],
                                 mem[moff[g]], b0[g] + f["p_t0_arr"][p], moff[g], (moff[g + 1] - moff[g]) * Gq,
                                 f["g_prows_arr"][g], int(g >= nsg)]
    assert f["p_desc"] % 4 == 0  # 16-byte aligned in the plan


def _softmax_state(qv, keys, vals):
    """(acc, m, l) of one query row over some tokens, natural-log domain."""
    s = keys @ qv
    m = s.max()
    w = np.exp(s - m)
    return w @ vals, m, w.sum()


def _row_warps(rows):
    return 1 if rows <= 8 else (2 if rows <= 16 else 4)


def _lanes(f, p, B, Gq):
    """The partial states piece p leaves: (record row offset of the lane,
    the piece's tiles it covers).  The tensor-core kernel leaves one state per
    row over all the piece's tiles; the CUDA-core kernel one per tile-lane
    that got a tile: tile t to lane (t + p) mod nl, lane tl's rows at record
    row tl * wr * 8 + row of the pass."""
    u = f["p_unit_arr"][p]
    g, ps = f["u_group_arr"][u], f["u_pass_arr"][u]
    moff = f["g_moff_arr"]
    rows = (moff[g + 1] - moff[g]) * Gq
    n = f["p_t1_arr"][p] - f["p_t0_arr"][p]
    if g < f["num_shared_groups"] and B in (16, 32, 64) and rows >= TC_MIN_ROWS:
        return [(0, list(range(n)))]
    pr = f["g_prows_arr"][g]
    wr = _row_warps(min(pr, rows - ps * pr))
    nl = 4 // wr
    out = []
    for tl in range(nl):
        ts = [t for t in range(n) if (t + p) % nl == tl]
        if ts:
            out.append((tl * wr * 8, ts))
    return out


def _emulate(f, q, kc, vc, tables, lens, scale):
    """The two steps of the shared decode, in float64, driven by the plan."""
    q, K, V = (x.double().numpy() for x in (q, kc, vc))
    tables, lens = tables.numpy(), lens.numpy()
    S, Hq, D = q.shape
    Hkv, B = K.shape[1], K.shape[2]
    Gq = Hq // Hkv
    moff, mem = f["g_moff_arr"], f["g_members_arr"]
    records = {}  # record index (piece * 32 + record row) -> (acc, m, l)
    for p in range(f["num_pieces"]):
        u = f["p_unit_arr"][p]
        g, kvh, ps = f["u_group_arr"][u], f["u_kvh_arr"][u], f["u_pass_arr"][u]
        members = mem[moff[g]:moff[g + 1]]
        first = f["g_b0_arr"][g] + f["p_t0_arr"][p]
        pr = f["g_prows_arr"][g]
        for off, ts in _lanes(f, p, B, Gq):
            keys, vals = [], []
            for t in ts:
                b = first + t
                ntok = min(B, int(lens[members[0]]) - b * B)  # a last block may be partly filled
                keys.append(K[tables[members[0], b], kvh][:ntok])
                vals.append(V[tables[members[0], b], kvh][:ntok])
            keys, vals = np.concatenate(keys), np.concatenate(vals)
            for r in range(ps * pr, min(ps * pr + pr, len(members) * Gq)):
                s, hh = members[r // Gq], r % Gq
                records[p * PASS_ROWS + off + r % pr] = _softmax_state(q[s, kvh * Gq + hh] * scale, keys, vals)
    out = np.zeros_like(q)
    roff, rrec = f["r_off_arr"], f["r_rec_arr"]
    assert len(roff) == S * Hq + 1
    for s in range(S):
        for h in range(Hq):
            kvh, hh = h // Gq, h % Gq
            want = []  # the row's records, from its memberships
            for k in range(f["s_moff_arr"][s], f["s_moff_arr"][s + 1]):
                g, mi = f["s_mgroup_arr"][k], f["s_midx_arr"][k]
                r = mi * Gq + hh
                pr = f["g_prows_arr"][g]
                u = f["g_ubase_arr"][g] + kvh * f["g_passes_arr"][g] + r // pr
                for p in range(f["u_poff_arr"][u], f["u_poff_arr"][u + 1]):
                    want += [p * PASS_ROWS + off + r % pr for off, _ in _lanes(f, p, B, Gq)]
            row = s * Hq + h
            got = [int(x) for x in rrec[roff[row]:roff[row + 1]]]
            assert got == want  # the merge's list of the row
            states = [records[x] for x in got]
            if states:
                M = max(m for _, m, _ in states)
                num = sum(a * np.exp(m - M) for a, m, _ in states)
                den = sum(l * np.exp(m - M) for _, m, l in states)
                out[s, h] = num / den
    return out


@pytest.mark.parametrize("name,nctas", [("prefix", 7), ("prefix", 304), ("longctx", 5), ("longctx4", 6), ("beam", 3)])
def test_plan_structure_and_emulated_decode_match_oracle(ops, name, nctas):
    q, kc, vc, tables, lens, scale = _case(name)
    B, Hq, Hkv = kc.shape[2], q.shape[1], kc.shape[1]
    plan = ops.share_plan(tables, lens, B, Hq, Hkv, nctas=nctas)
    f = ops.plan_fields(plan)
    assert f["num_groups"] > 0
    _check_structure(f, tables.numpy(), lens.numpy(), B, Hq, Hkv)
    got = _emulate(f, q, kc, vc, tables, lens, scale)
    ref = reference.decode(q, kc, vc, tables.numpy(), lens.numpy(), scale)
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)


def test_plan_of_unshared_tables_has_no_groups(ops):
    inp = W.make_inputs(W.scaled(W.GQA, num_seqs=4, num_blocks=4 * 256 + 3), 0)
    plan = ops.share_plan(inp.block_tables, inp.context_lens, 16, 32, 8, nctas=11)
    f = ops.plan_fields(plan)
    assert f["num_shared_groups"] == 0 and f["num_groups"] == 4  # each sequence's own group only
    assert list(f["s_start_arr"]) == [0] * 4
    assert f["own_tiles"] == 1
    _check_structure(f, inp.block_tables.numpy(), inp.context_lens.numpy(), 16, 32, 8)


def test_plan_edge_cases(ops):
    # identical tables: one group over all full blocks; the partial tail, an
    # empty sequence and a one-token sequence stay private
    B = 16
    row = list(range(10))
    tables = torch.tensor([row, row, row, row], dtype=torch.int32)
    lens = torch.tensor([150, 150, 0, 7], dtype=torch.int32)  # 9 full blocks + 6 tokens
    f = ops.plan_fields(ops.share_plan(tables, lens, B, 4, 2, nctas=3))
    assert f["num_shared_groups"] == 1 and f["num_groups"] == 4  # one shared, three own groups
    assert list(f["g_members_arr"][:2]) == [0, 1] and (f["g_b0_arr"][0], f["g_b1_arr"][0]) == (0, 9)
    assert list(f["g_members_arr"][2:]) == [0, 1, 3]  # the partial tails, and the one-token sequence
    assert list(f["s_start_arr"]) == [9, 9, 0, 0]
    assert f["own_tiles"] == 1
    _check_structure(f, tables.numpy(), lens.numpy(), B, 4, 2)
    # 40 members x 4 heads = 160 rows: 5 passes per kv head
    tables = torch.tensor([row] * 40, dtype=torch.int32)
    lens = torch.full((40,), 64, dtype=torch.int32)
    f = ops.plan_fields(ops.share_plan(tables, lens, B, 8, 2, nctas=9))
    assert f["num_groups"] == 1 and f["g_passes_arr"][0] == 5 and f["num_units"] == 10
    assert list(f["s_start_arr"]) == [4] * 40  # every block shared: nothing of their own
    assert f["own_tiles"] == 0 and f["num_shared_groups"] == 1  # no own group
    # 160 rows per kv head: the tensor cores take it, two 128-row items per kv head
    assert f["num_tc_items"] == 4 and f["c_poff_arr"][-1] == 0
    _check_structure(f, tables.numpy(), lens.numpy(), B, 8, 2)
    # with a block size that does not divide a 64-token step it stays on the CUDA cores
    f = ops.plan_fields(ops.share_plan(tables, lens, 48, 8, 2, nctas=9))
    assert f["num_tc_items"] == 0


def test_plan_rejects_bad_arguments_and_small_buffers(ops):
    import ctypes

    tables = torch.zeros(2, 4, dtype=torch.int32)
    lens = torch.tensor([16, 16], dtype=torch.int32)
    need = ctypes.c_size_t(0)
    assert ops.lib.pa_share_plan(tables.data_ptr(), 4, lens.data_ptr(), 2, 16, 6, 4, 8, None, 0,
                                 ctypes.byref(need)) == 1  # heads not a multiple of kv heads
    assert ops.lib.pa_share_plan(tables.data_ptr(), 4, lens.data_ptr(), 2, 16, 8, 4, 8, None, 0,
                                 ctypes.byref(need)) == 0
    small = torch.zeros(int(need.value) - 1, dtype=torch.int32)
    assert ops.lib.pa_share_plan(tables.data_ptr(), 4, lens.data_ptr(), 2, 16, 8, 4, 8, small.data_ptr(),
                                 small.numel(), ctypes.byref(need)) == 4  # PA_ERR_WORKSPACE
