"""Decode parity under the contiguous allocation policy.

cf-1.com news/5879632, section 5.1, suggests keeping a sequence's blocks
physically together so that reads stay linear.  Here the block tables come from
``BlockManager(policy="contiguous")`` (with frees and re-allocations in between,
so some sequences are split into several runs) and from the workloads'
``placement="contiguous"``.  The step (``pa_write_decode``: each sequence's new
token written at position L - 1, then the decode) must match the oracle, and
give bit-identical output and pools to the same logical data under a random
relabelling of the physical blocks: the decode's arithmetic depends only on
logical positions, never on where a block sits.
"""
import numpy as np
import pytest
import torch

from gpu_utils import assert_attention_close, oracle_step
from paged_kv_cache_170_gb300 import workloads as W
from paged_kv_cache_170_gb300.block_manager import BlockManager

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


def manager_case(seed, S, Hq, Hkv, D, B, dtype, max_len):
    """A decode step whose tables a contiguous-policy manager built: S
    sequences prefilled, every third freed and replaced by a longer one (so
    the pool is fragmented), then one new token appended to each."""
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(1, max_len, (S,), generator=g).tolist()
    width = -(-(max_len + max_len // 2 + 1) // B)
    NB = S * width + 8
    mgr = BlockManager(NB, B, policy="contiguous")
    seqs = list(range(S))
    for s in seqs:
        mgr.allocate(s, lens[s])
    for s in seqs[::3]:
        mgr.free_seq(s)
    for s in seqs[::3]:
        lens[s] = min(lens[s] + int(torch.randint(1, max_len // 2, (1,), generator=g)), width * B - 1)
        mgr.allocate(s, lens[s])
    slots = [mgr.append_slot(s)[0] for s in seqs]
    mgr.check()
    tables = torch.from_numpy(mgr.block_tables(seqs, width=width))
    ctx = torch.from_numpy(mgr.context_lens(seqs))
    kc = W.randn((NB, Hkv, B, D), dtype, g)
    vc = W.randn((NB, Hkv, B, D), dtype, g)
    q = W.randn((S, Hq, D), dtype, g)
    nk = W.randn((S, Hkv, D), dtype, g)
    nv = W.randn((S, Hkv, D), dtype, g)
    w = W.scaled(W.GQA, name="manager", num_seqs=S, num_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=B,
                 dtype=dtype, num_blocks=NB, max_blocks_per_seq=width, placement="contiguous")
    inp = W.DecodeInputs(w, q, kc, vc, tables, ctx, nk, nv, torch.arange(S, dtype=torch.int32),
                         (ctx - 1).to(torch.int32), torch.zeros((0, 2), dtype=torch.int64), float(D) ** -0.5)
    return inp, np.asarray(slots, dtype=np.int64)


def consecutive_fraction(tables, lens, B):
    """Share of a step's adjacent (block i, block i + 1) table pairs that are
    consecutive physical ids."""
    hit = tot = 0
    for row, L in zip(tables.tolist(), lens.tolist()):
        n = -(-L // B)
        for i in range(n - 1):
            tot += 1
            hit += row[i + 1] == row[i] + 1
    return hit / max(tot, 1)


def write_decode(ops, inp):
    err = ops.new_error_word(DEV)
    out = ops.pa_write_decode(inp.q, inp.new_key, inp.new_value, inp.k_cache, inp.v_cache, inp.block_tables,
                              inp.context_lens, inp.scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, ops.error_names(int(err.item()))
    return out


def relabel(inp, seed):
    """The same logical data with physical block p moved to pi[p]."""
    NB = inp.k_cache.shape[0]
    pi = torch.randperm(NB, generator=torch.Generator().manual_seed(seed))
    k2, v2 = torch.empty_like(inp.k_cache), torch.empty_like(inp.v_cache)
    k2[pi] = inp.k_cache
    v2[pi] = inp.v_cache
    t2 = torch.where(inp.block_tables >= 0, pi.to(torch.int32)[inp.block_tables.clamp(min=0).long()],
                     inp.block_tables)
    other = W.DecodeInputs(inp.workload, inp.q, k2, v2, t2, inp.context_lens, inp.new_key, inp.new_value,
                           inp.new_seq, inp.new_pos, inp.copy_pairs, inp.scale)
    return other, pi


@pytest.mark.parametrize("case", ["gqa_bf16", "mha_f16", "longblock_bf16"])
def test_contiguous_manager_tables_match_oracle_and_random_placement(ops, case):
    S, Hq, Hkv, D, B, dtype, max_len = {
        "gqa_bf16": (12, 32, 8, 128, 16, torch.bfloat16, 3000),
        "mha_f16": (8, 16, 16, 128, 16, torch.float16, 1500),
        "longblock_bf16": (6, 16, 2, 64, 32, torch.bfloat16, 2500),
    }[case]
    cpu, mgr_slots = manager_case(5, S, Hq, Hkv, D, B, dtype, max_len)
    assert consecutive_fraction(cpu.block_tables, cpu.context_lens, B) > 0.9
    slots_ref, kc_ref, vc_ref, out_ref = oracle_step(cpu)
    assert np.array_equal(slots_ref, mgr_slots)  # the manager's slots are the table lookup's

    inp = cpu.to(DEV)
    out = write_decode(ops, inp)
    assert torch.equal(inp.k_cache.cpu(), kc_ref) and torch.equal(inp.v_cache.cpu(), vc_ref)
    assert_attention_close(out, out_ref, strict=True)

    scattered, pi = relabel(cpu, seed=17)
    assert consecutive_fraction(scattered.block_tables, scattered.context_lens, B) < 0.1
    inp2 = scattered.to(DEV)
    out2 = write_decode(ops, inp2)
    assert torch.equal(out2, out)
    assert torch.equal(inp2.k_cache.cpu()[pi], kc_ref) and torch.equal(inp2.v_cache.cpu()[pi], vc_ref)


@pytest.mark.parametrize("name", ["gqa", "mha"])
def test_contiguous_workload_placement_through_the_bench_step(ops, name):
    """The benchmark's step (CUDA graphs, pa_write_decode) on a scaled copy of
    the workload with placement="contiguous"."""
    from paged_kv_cache_170_gb300.step import DecodeStep

    base = W.WORKLOADS[name]
    w = W.scaled(base, num_seqs=10, num_blocks=10 * base.max_blocks_per_seq + 3, placement="contiguous")
    cpu = W.make_inputs(w, seed=2)
    assert consecutive_fraction(cpu.block_tables, cpu.context_lens, w.block_size) == 1.0
    slots_ref, kc_ref, vc_ref, out_ref = oracle_step(cpu)
    inp = cpu.to(DEV)
    runner = DecodeStep(inp)  # its construction runs the step once eagerly, then records the graphs
    torch.cuda.synchronize()
    assert runner.fused and int(runner.err.item()) == 0
    assert torch.equal(inp.k_cache.cpu(), kc_ref) and torch.equal(inp.v_cache.cpu(), vc_ref)
    assert_attention_close(runner.out, out_ref, strict=True)
    first = runner.out.clone()
    runner.run()  # a graph replay rewrites the same rows and gives the same output
    torch.cuda.synchronize()
    assert torch.equal(runner.out, first)
