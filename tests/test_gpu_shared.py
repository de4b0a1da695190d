"""pa_decode_shared: the decode that reads each shared block once per group of
sharers (plan from pa_share_plan), against the float64 oracle, on the
shared-prefix and long-context workloads (small and full size), a nested
beam-like trie, and edge cases.  It must also agree with pa_decode."""
import math

import numpy as np
import pytest
import torch

from gpu_utils import assert_attention_close, oracle_step
from oracle import native
from paged_kv_cache_170_gb300 import scenarios
from paged_kv_cache_170_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_170_gb300 import build

    build.build()
    from paged_kv_cache_170_gb300 import ops as _ops

    return _ops


def _pre_step(ops, inp):
    """The step's copies, slot lookup and writes (the state the decode reads)."""
    err = ops.new_error_word(inp.q.device)
    if inp.copy_pairs.numel():
        ops.pa_copy_blocks(inp.k_cache, inp.v_cache, inp.copy_pairs, err)
    if inp.new_seq.numel():
        slots = ops.pa_slot_mapping(inp.block_tables, inp.new_seq, inp.new_pos, inp.k_cache.shape[2],
                                    inp.k_cache.shape[0], None, err)
        ops.pa_write_kv(inp.new_key, inp.new_value, inp.k_cache, inp.v_cache, slots, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0


def _shared(ops, q, kc, vc, tables, lens, scale, workspace=None):
    plan = ops.share_plan(tables, lens, kc.shape[2], q.shape[1], kc.shape[1])
    plan_dev = plan.to(q.device)
    err = ops.new_error_word(q.device)
    out = ops.pa_decode_shared(q, kc, vc, tables, lens, scale, plan, plan_dev, workspace=workspace, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, ops.error_names(int(err.item()))
    return out, ops.plan_fields(plan)


def _small(name, seed=0):
    if name == "prefix":
        return scenarios.shared_prefix_inputs(seed, num_parents=4, prefix_tokens=256, suffix_max=300,
                                              w=W.scaled(W.PREFIX, num_blocks=300, max_blocks_per_seq=40))
    if name == "longctx":
        return scenarios.long_context_inputs(seed, num_prompts=2, branches=3, prompt_tokens=2048, suffix_max=200,
                                             w=W.scaled(W.LONGCTX, num_blocks=200, max_blocks_per_seq=80))
    if name == "prefix_wide":  # 20 sharers x 4 heads = 80 rows: three passes per kv head
        return scenarios.shared_prefix_inputs(seed, num_parents=10, prefix_tokens=320, suffix_max=100,
                                              w=W.scaled(W.PREFIX, num_blocks=400, max_blocks_per_seq=40))
    raise KeyError(name)


@pytest.mark.parametrize("name", ["prefix", "longctx", "prefix_wide"])
def test_shared_decode_small_matches_oracle_and_plain_decode(ops, name):
    cpu = _small(name)
    inp = cpu.to(DEV)
    _pre_step(ops, inp)
    out, f = _shared(ops, inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale)
    assert f["num_groups"] > 0
    _, _, _, ref = oracle_step(cpu)
    assert_attention_close(out, ref, strict=True)
    plain = ops.pa_decode(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale)
    torch.cuda.synchronize()
    assert (out.float() - plain.float()).abs().max().item() <= 4e-3


@pytest.mark.parametrize("name,sample", [("prefix", None), ("longctx", [0, 3, 6, 13, 22, 31])])
def test_shared_decode_full_size(ops, name, sample):
    inp = scenarios.shared_prefix_inputs(0, device=DEV) if name == "prefix" else \
        scenarios.long_context_inputs(0, device=DEV)
    cpu = inp.to("cpu")
    _pre_step(ops, inp)
    out, f = _shared(ops, inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale)
    assert f["num_groups"] > 0
    _, _, _, ref = oracle_step(cpu, seqs=sample)
    got = out if sample is None else out[torch.as_tensor(sample, device=out.device)]
    print(name, assert_attention_close(got, ref, strict=True), "groups", f["num_groups"], "pieces", f["num_pieces"])


def _random_pool(S, Hq, Hkv, D, B, NB, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(S, Hq, D, generator=g).to(dtype)
    kc = torch.randn(NB, Hkv, B, D, generator=g).to(dtype)
    vc = torch.randn(NB, Hkv, B, D, generator=g).to(dtype)
    return q, kc, vc


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_shared_decode_edge_cases(ops, dtype):
    """Identical tables with a partial tail, an empty sequence, a sequence
    shorter than one block, a sequence whose blocks are all shared, and a
    sequence outside every group; then sequences with no blocks of their own
    at all; head_dim 64 and 128."""
    for D in (64, 128):
        S, Hq, Hkv, B, NB = 6, 8, 2, 16, 64
        q, kc, vc = _random_pool(S, Hq, Hkv, D, B, NB, dtype, seed=D)
        row = list(range(10))
        tables = torch.tensor([row, row, row, row, row, list(range(20, 30))], dtype=torch.int32)
        lens = torch.tensor([150, 150, 0, 7, 144, 150], dtype=torch.int32)
        scale = 1.0 / math.sqrt(D)
        args = [x.to(DEV) for x in (q, kc, vc, tables, lens)]
        out, f = _shared(ops, *args, scale)
        assert f["num_groups"] >= 1
        ref = native.decode(q, kc, vc, tables.numpy(), lens.numpy(), scale)
        assert_attention_close(out, ref, strict=False)
        assert torch.count_nonzero(out[2]) == 0  # empty sequence: zero row
        # every sequence's blocks all shared and full: no own group, no own tiles
        full = torch.tensor([row] * 4, dtype=torch.int32)
        lens_full = torch.full((4,), 144, dtype=torch.int32)
        out, f = _shared(ops, q[:4].to(DEV), args[1], args[2], full.to(DEV), lens_full.to(DEV), scale)
        assert f["num_groups"] == 1 and f["own_tiles"] == 0
        ref = native.decode(q[:4], kc, vc, full.numpy(), lens_full.numpy(), scale)
        assert_attention_close(out, ref, strict=False)


@pytest.mark.parametrize("B", [16, 32])
def test_shared_decode_own_groups_of_two_passes(ops, B):
    """16 query heads per kv head: a sequence's own blocks are read in two
    8-row passes; partly filled last blocks of every length mod B."""
    S, Hq, Hkv, D = 6, 32, 2, 128
    NB = 80
    q, kc, vc = _random_pool(S, Hq, Hkv, D, B, NB, torch.bfloat16, seed=B)
    shared = list(range(4))
    tables = torch.tensor([shared + list(range(10 + 8 * i, 18 + 8 * i)) for i in range(S)], dtype=torch.int32)
    lens = torch.tensor([4 * B + 1, 4 * B + B - 1, 6 * B, 5 * B + 7, 4 * B, 2 * B + 3], dtype=torch.int32)
    scale = 1.0 / math.sqrt(D)
    out, f = _shared(ops, *[x.to(DEV) for x in (q, kc, vc, tables, lens)], scale)
    assert f["num_shared_groups"] >= 1 and f["num_groups"] > f["num_shared_groups"]
    ref = native.decode(q, kc, vc, tables.numpy(), lens.numpy(), scale)
    assert_attention_close(out, ref, strict=False)


@pytest.mark.parametrize("B,D,dtype,members,Hq,Hkv,run", [
    (16, 128, torch.bfloat16, 40, 8, 2, 37),   # 160 rows: two 128-row items, a short last step
    (32, 64, torch.float16, 12, 16, 2, 21),    # 96 rows, two blocks per step
    (64, 128, torch.bfloat16, 9, 32, 8, 7),    # 36 rows, one block per step
    (16, 64, torch.bfloat16, 8, 32, 8, 64),    # exactly 32 rows, a run of 16 whole steps
    (16, 128, torch.float16, 40, 8, 8, 23),    # one query head per kv head (G = 1): 40 rows
    (32, 128, torch.bfloat16, 4, 64, 4, 11),   # G = 16: a member's 16 heads fill half a pass
])
def test_shared_decode_tensor_core_groups(ops, B, D, dtype, members, Hq, Hkv, run):
    """Groups with 32 or more query rows per kv head are computed on the
    tensor cores (the prompt kernel's pipeline over the group's rows): every
    block size it takes, both head dims and dtypes, row counts that are not a
    multiple of 128, runs that end in a short step; some members also have
    blocks of their own with a partly filled last one."""
    S = members + 2
    own = [0, 3, 1, 0, 2] * ((S + 4) // 5)
    NB = run + sum(own[:S]) + 2 * 5 + 4
    q, kc, vc = _random_pool(S, Hq, Hkv, D, B, NB, dtype, seed=B + D + members)
    tables = torch.full((S, run + 6), 0, dtype=torch.int32)
    lens = torch.zeros(S, dtype=torch.int32)
    nxt = run
    for s in range(S):
        if s < members:  # the shared run, then own blocks (the last one partly filled)
            tables[s, :run] = torch.arange(run, dtype=torch.int32)
            k = own[s]
            tables[s, run:run + k] = torch.arange(nxt, nxt + k, dtype=torch.int32)
            nxt += k
            lens[s] = run * B + (k - 1) * B + 1 + s % B if k else run * B
        else:  # two sequences outside every group
            tables[s, :5] = torch.arange(nxt, nxt + 5, dtype=torch.int32)
            nxt += 5
            lens[s] = 4 * B + 3
    scale = 1.0 / math.sqrt(D)
    out, f = _shared(ops, *[x.to(DEV) for x in (q, kc, vc, tables, lens)], scale)
    assert f["num_tc_items"] > 0
    ref = native.decode(q, kc, vc, tables.numpy(), lens.numpy(), scale)
    assert_attention_close(out, ref, strict=False)
    plain = ops.pa_decode(*[x.to(DEV) for x in (q, kc, vc, tables, lens)], scale)
    torch.cuda.synchronize()
    assert (out.float() - plain.float()).abs().max().item() <= 4e-3


def test_shared_decode_deterministic_reusable_workspace_and_no_group_plan(ops):
    cpu = _small("prefix", seed=1)
    inp = cpu.to(DEV)
    _pre_step(ops, inp)
    plan = ops.share_plan(inp.block_tables, inp.context_lens, 16, inp.q.shape[1], inp.k_cache.shape[1])
    ws = ops.new_shared_workspace(plan, inp.q.shape[0], inp.q.shape[1], inp.k_cache.shape[1], inp.q.shape[2], DEV)
    pd = plan.to(DEV)
    a = ops.pa_decode_shared(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale, plan,
                             pd, workspace=ws).clone()
    b = ops.pa_decode_shared(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale, plan,
                             pd, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    # tables without sharing: the plan has no groups and the call is pa_decode
    g = W.make_inputs(W.scaled(W.GQA, num_seqs=3, num_blocks=3 * 256 + 5), 0).to(DEV)
    out, f = _shared(ops, g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale)
    assert f["num_shared_groups"] == 0
    plain = ops.pa_decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale)
    torch.cuda.synchronize()
    assert torch.equal(out, plain)


def test_shared_decode_rejects_fp32_and_mismatched_plans(ops):
    q, kc, vc = _random_pool(2, 4, 2, 64, 16, 8, torch.float32, seed=0)
    tables = torch.tensor([[0, 1], [0, 1]], dtype=torch.int32)
    lens = torch.tensor([32, 32], dtype=torch.int32)
    plan = ops.share_plan(tables, lens, 16, 4, 2)
    with pytest.raises(ops.PagedKVError, match="UNSUPPORTED"):
        ops.pa_decode_shared(q.to(DEV), kc.to(DEV), vc.to(DEV), tables.to(DEV), lens.to(DEV), 0.1, plan,
                             plan.to(DEV))
    q16 = q.to(torch.bfloat16).to(DEV)
    other = ops.share_plan(tables, lens, 16, 8, 2)  # built for 8 query heads
    with pytest.raises(ops.PagedKVError, match="INVALID"):
        ops.pa_decode_shared(q16, kc.to(torch.bfloat16).to(DEV), vc.to(torch.bfloat16).to(DEV), tables.to(DEV),
                             lens.to(DEV), 0.1, other, other.to(DEV), workspace=torch.zeros(1 << 22,
                                                                                             dtype=torch.uint8,
                                                                                             device=DEV))
