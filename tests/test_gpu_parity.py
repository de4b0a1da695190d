"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bit-exact: slot lookup, K/V write, copy-on-write copies, and the decode
output's invariance under block relabelling / sharing.  Attention output:
fp16/bf16 max abs <= 2e-3 and max rel <= 1e-2 (over |ref| >= 1e-2) on the
workloads; fp32 abs 1e-5 + rel 1e-4.
"""
import numpy as np
import pytest
import torch

from gpu_utils import assert_attention_close, oracle_step, valid_blocks
from oracle import native
from paged_kv_cache_170_gb300 import scenarios
from paged_kv_cache_170_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_170_gb300 import build

    build.build()
    from paged_kv_cache_170_gb300 import ops as _ops

    return _ops


DEV = "cuda"


def small_case(name, seed=0):
    if name == "tiny":
        return W.make_inputs(W.TINY, seed)
    if name == "mha_small":
        return W.make_inputs(W.scaled(W.MHA, num_seqs=6, num_blocks=900), seed)
    if name == "gqa_small":
        return W.make_inputs(W.scaled(W.GQA, num_seqs=3, num_blocks=3 * 256 + 17), seed)
    if name == "prefix_small":
        return scenarios.shared_prefix_inputs(seed, num_parents=4, prefix_tokens=256, suffix_max=300,
                                              w=W.scaled(W.PREFIX, num_blocks=300, max_blocks_per_seq=40))
    if name == "longctx_small":
        return scenarios.long_context_inputs(seed, num_prompts=2, branches=3, prompt_tokens=2048, suffix_max=200,
                                             w=W.scaled(W.LONGCTX, num_blocks=200, max_blocks_per_seq=80))
    raise KeyError(name)


def run_step(ops, inp):
    err = ops.new_error_word(inp.q.device)
    slots = torch.empty(inp.new_seq.numel(), dtype=torch.int64, device=inp.q.device)
    out = ops.decode_step(inp, slots=slots, err=err)
    torch.cuda.synchronize()
    return out, slots, int(err.item())


@pytest.mark.parametrize("name", ["tiny", "mha_small", "gqa_small", "prefix_small", "longctx_small"])
def test_step_parity_small(ops, name):
    cpu = small_case(name)
    inp = cpu.to(DEV)
    out, slots, err = run_step(ops, inp)
    assert err == 0, ops.error_names(err)
    slots_ref, kc_ref, vc_ref, out_ref = oracle_step(cpu)
    assert np.array_equal(slots.cpu().numpy(), slots_ref)
    if "manager_slots" in cpu.extra:
        assert np.array_equal(cpu.extra["manager_slots"].numpy(), slots_ref)
    assert torch.equal(inp.k_cache.cpu(), kc_ref) and torch.equal(inp.v_cache.cpu(), vc_ref)
    assert_attention_close(out, out_ref, strict=True)


def _full_case(name, seed=0):
    if name == "gqa":
        return W.make_inputs(W.GQA, seed, device=DEV)
    if name == "mha":
        return W.make_inputs(W.MHA, seed, device=DEV)
    if name == "prefix":
        return scenarios.shared_prefix_inputs(seed, device=DEV)
    if name == "longctx":
        return scenarios.long_context_inputs(seed, device=DEV)
    raise KeyError(name)


@pytest.mark.parametrize("name,sample", [("gqa", None), ("mha", None), ("prefix", None),
                                         ("longctx", [0, 5, 10, 15, 21, 31])])
def test_step_parity_full_size(ops, name, sample):
    """Full-size workload, the same calls the benchmark times; the oracle checks
    every sequence (or the listed sample for the long-context workload)."""
    inp = _full_case(name)
    cpu = inp.to("cpu")  # state before the step
    out, slots, err = run_step(ops, inp)
    assert err == 0, ops.error_names(err)
    slots_ref, kc_ref, vc_ref, out_ref = oracle_step(cpu, seqs=sample)
    assert np.array_equal(slots.cpu().numpy(), slots_ref)
    assert torch.equal(inp.k_cache.cpu(), kc_ref) and torch.equal(inp.v_cache.cpu(), vc_ref)
    got = out if sample is None else out[torch.as_tensor(sample, device=out.device)]
    stats = assert_attention_close(got, out_ref, strict=True)
    print(name, stats)


# ------------------------------------------------------------------ generic cases
def random_case(lens, Hq, Hkv, D, B, dtype, seed=0, pad_tables=False, extra_blocks=5):
    g = torch.Generator().manual_seed(seed)
    S = len(lens)
    nbl = valid_blocks(lens, B)
    width = max(max(nbl) if nbl else 0, 1)
    NB = sum(nbl) + extra_blocks + (0 if pad_tables else S * width)
    perm = torch.randperm(NB, generator=g)
    tables = torch.full((S, width), -1, dtype=torch.int32)
    k = 0
    for s in range(S):
        n = nbl[s] if pad_tables else width
        tables[s, :n] = perm[k:k + n].to(torch.int32)
        k += n
    kc = W.randn((NB, Hkv, B, D), dtype, g)
    vc = W.randn((NB, Hkv, B, D), dtype, g)
    q = W.randn((S, Hq, D), dtype, g)
    lens_t = torch.tensor(lens, dtype=torch.int32)
    return q, kc, vc, tables, lens_t


EDGE = {
    # name: (lens, Hq, Hkv, D, B, dtype, pad_tables)
    "zero_one_tails": ([0, 1, 0, 2, 16, 17, 31, 33], 8, 2, 128, 16, torch.bfloat16, True),
    "block1_fp16": ([5, 33, 1], 4, 4, 64, 1, torch.float16, False),
    "block64_bf16": ([1, 64, 65, 200], 8, 8, 128, 64, torch.bfloat16, True),
    "group3": ([7, 100, 257], 6, 2, 128, 16, torch.bfloat16, False),
    "group6": ([50, 9], 12, 2, 64, 8, torch.float16, True),
    "group16": ([300, 45, 1], 32, 2, 128, 32, torch.bfloat16, True),
    "group8_d64": ([77, 500], 16, 2, 64, 16, torch.bfloat16, False),
    "one_long_sequence": ([50000], 8, 1, 128, 16, torch.bfloat16, True),
    "fp32_d128_b8": ([3, 130, 64, 0, 9], 4, 2, 128, 8, torch.float32, True),
    "fp32_b64_d128": ([70, 129], 2, 1, 128, 64, torch.float32, True),
}


@pytest.mark.parametrize("name", sorted(EDGE))
def test_decode_edge_cases(ops, name):
    lens, Hq, Hkv, D, B, dtype, pad = EDGE[name]
    q, kc, vc, tables, lens_t = random_case(lens, Hq, Hkv, D, B, dtype, seed=len(name), pad_tables=pad)
    scale = D ** -0.5
    err = ops.new_error_word(DEV)
    out = ops.pa_decode(q.to(DEV), kc.to(DEV), vc.to(DEV), tables.to(DEV), lens_t.to(DEV), scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, ops.error_names(int(err.item()))
    ref = native.decode(q, kc, vc, tables.numpy(), lens_t.numpy(), scale)
    assert_attention_close(out, ref, strict=False)
    for s, L in enumerate(lens):
        if L == 0:
            assert torch.count_nonzero(out[s]) == 0


def test_many_short_sequences(ops):
    g = torch.Generator().manual_seed(3)
    lens = torch.randint(0, 41, (2000,), generator=g).tolist()
    q, kc, vc, tables, lens_t = random_case(lens, 4, 4, 64, 16, torch.float16, seed=9, pad_tables=True)
    out = ops.pa_decode(q.to(DEV), kc.to(DEV), vc.to(DEV), tables.to(DEV), lens_t.to(DEV), 0.125)
    ref = native.decode(q, kc, vc, tables.numpy(), lens_t.numpy(), 0.125)
    assert_attention_close(out, ref, strict=False)


@pytest.mark.parametrize("case", ["long_among_short", "one_tile_segments_few_ctas"])
def test_cost_weighted_split(ops, case):
    """CTA ranges split tiles + a fixed cost per (sequence, head) segment:
    long sequences among many one-to-three-block ones (boundaries shift with
    the short segments; long pairs are cut among several CTAs), and one-tile
    segments whose total cost is below the CTA count (some CTAs own only
    fixed-cost positions, i.e. no tile)."""
    g = torch.Generator().manual_seed(21)
    if case == "long_among_short":
        lens = torch.randint(1, 48, (300,), generator=g).tolist()
        for i in range(0, 300, 37):
            lens[i] = int(torch.randint(2000, 6000, (1,), generator=g))
        Hq = Hkv = 16
    else:
        lens = [1] * 10 + [0, 3]
        Hq, Hkv = 8, 4
    q, kc, vc, tables, lens_t = random_case(lens, Hq, Hkv, 128, 16, torch.float16, seed=22, pad_tables=True)
    err = ops.new_error_word(DEV)
    out = ops.pa_decode(q.to(DEV), kc.to(DEV), vc.to(DEV), tables.to(DEV), lens_t.to(DEV), 0.09, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, ops.error_names(int(err.item()))
    ref = native.decode(q, kc, vc, tables.numpy(), lens_t.numpy(), 0.09)
    assert_attention_close(out, ref, strict=False)


def test_relabelled_blocks_give_bit_identical_output(ops):
    q, kc, vc, tables, lens = random_case([300, 4096, 17, 1000], 32, 8, 128, 16, torch.bfloat16, seed=1)
    args = [t.to(DEV) for t in (q, kc, vc, tables, lens)]
    a = ops.pa_decode(*args, 0.088)
    pi = torch.randperm(kc.shape[0], generator=torch.Generator().manual_seed(2))
    k2, v2 = torch.empty_like(kc), torch.empty_like(vc)
    k2[pi] = kc
    v2[pi] = vc
    t2 = pi.to(torch.int32)[tables.long()]
    b = ops.pa_decode(args[0], k2.to(DEV), v2.to(DEV), t2.to(DEV), args[4], 0.088)
    assert torch.equal(a, b)


def test_shared_layout_equals_private_copies_bit_exact(ops):
    cpu = small_case("prefix_small", seed=4)
    inp = cpu.to(DEV)
    out, _, err = run_step(ops, inp)
    assert err == 0
    # give every sequence private copies of all its blocks
    k, v = inp.k_cache.cpu(), inp.v_cache.cpu()
    tables = inp.block_tables.cpu()
    lens = inp.context_lens.cpu()
    nbl = valid_blocks(lens.tolist(), k.shape[2])
    total = sum(nbl)
    kp = torch.empty((total,) + tuple(k.shape[1:]), dtype=k.dtype)
    vp = torch.empty_like(kp)
    tp = torch.full_like(tables, -1)
    i = 0
    for s, n in enumerate(nbl):
        for bidx in range(n):
            kp[i] = k[tables[s, bidx]]
            vp[i] = v[tables[s, bidx]]
            tp[s, bidx] = i
            i += 1
    again = ops.pa_decode(inp.q, kp.to(DEV), vp.to(DEV), tp.to(DEV), inp.context_lens, inp.scale)
    assert torch.equal(out, again)


def test_decode_is_deterministic_and_workspace_reusable(ops):
    # the workspace's counters are back at zero after every call, so one
    # workspace serves calls of different shapes; results do not change
    ws = None
    outs = []
    for name in ("mha_small", "gqa_small", "mha_small"):
        inp = small_case(name, seed=7).to(DEV)
        if ws is None:
            ws = ops.new_workspace(4096, 64, 1, 128, DEV)
        outs.append(ops.pa_decode(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale,
                                  workspace=ws))
        assert torch.count_nonzero(ws[-(4096 * 64 * 4):]) == 0
    assert torch.equal(outs[0], outs[2])


def test_one_workspace_serves_calls_of_any_shape(ops):
    """Calls of different head dims, group sizes, dtypes and block sizes share
    one workspace and each gives the bits a fresh workspace gives: the
    counters sit at the same offset for every shape, and every call leaves
    them at zero."""
    shapes = [  # (D, Hq, Hkv, B, dtype)
        (64, 8, 1, 16, torch.float16),
        (128, 32, 8, 16, torch.bfloat16),
        (64, 16, 2, 32, torch.bfloat16),
        (128, 16, 2, 8, torch.float16),  # block size not a multiple of 16: the CUDA-core kernel
        (128, 8, 8, 16, torch.float16),
        (64, 8, 1, 16, torch.float16),
    ]
    ws = ops.new_workspace(64, 32, 1, 128, DEV)
    for i, (D, Hq, Hkv, B, dtype) in enumerate(shapes):
        q, kc, vc, tables, lens = random_case([700, 33, 1500, 0, 260, 4000, 17], Hq, Hkv, D, B, dtype, seed=i)
        args = [x.to(DEV) for x in (q, kc, vc, tables, lens)]
        got = ops.pa_decode(*args, 0.08, workspace=ws)
        fresh = ops.pa_decode(*args, 0.08)
        torch.cuda.synchronize()
        assert torch.equal(got, fresh), (D, Hq, Hkv, B, dtype)
        assert torch.count_nonzero(ws[-(64 * 32 * 4):]) == 0


def test_device_bounds_checks_raise_error_bits(ops):
    q, kc, vc, tables, lens = random_case([40, 20], 4, 2, 128, 16, torch.bfloat16, seed=5, pad_tables=True)
    NB = kc.shape[0]
    q, kc, vc, lens = q.to(DEV), kc.to(DEV), vc.to(DEV), lens.to(DEV)
    bad = tables.clone()
    bad[0, 1] = NB + 3
    err = ops.new_error_word(DEV)
    ops.pa_decode(q, kc, vc, bad.to(DEV), lens, 0.1, err=err)
    torch.cuda.synchronize()
    assert "BLOCK_ID" in ops.error_names(int(err.item()))
    err.zero_()
    ops.pa_decode(q, kc, vc, tables.to(DEV), torch.tensor([40, 20 + 16 * 5], dtype=torch.int32, device=DEV), 0.1,
                  err=err)
    torch.cuda.synchronize()
    assert "CONTEXT" in ops.error_names(int(err.item()))
    err.zero_()
    key = torch.zeros(2, 2, 128, dtype=torch.bfloat16, device=DEV)
    ops.pa_write_kv(key, key, kc, vc, torch.tensor([3, NB * 16], dtype=torch.int64, device=DEV), err=err)
    torch.cuda.synchronize()
    assert ops.error_names(int(err.item())) == ["SLOT"]
    err.zero_()
    ops.pa_slot_mapping(tables.to(DEV), torch.tensor([0, 1], dtype=torch.int32, device=DEV),
                        torch.tensor([5, 1000], dtype=torch.int32, device=DEV), 16, NB, err=err)
    torch.cuda.synchronize()
    assert ops.error_names(int(err.item())) == ["POSITION"]
    err.zero_()
    ops.pa_copy_blocks(kc, vc, torch.tensor([[0, NB]], dtype=torch.int64, device=DEV), err=err)
    torch.cuda.synchronize()
    assert ops.error_names(int(err.item())) == ["BLOCK_ID"]


def test_host_validation(ops):
    inp = small_case("tiny").to(DEV)
    small = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(ops.PagedKVError, match="WORKSPACE"):
        ops.pa_decode(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, 0.1, workspace=small)
    k96 = torch.zeros(4, 1, 4, 96, device=DEV)
    with pytest.raises(ops.PagedKVError, match="UNSUPPORTED"):
        ops.pa_decode(torch.zeros(1, 1, 96, device=DEV), k96, k96, torch.zeros(1, 1, dtype=torch.int32, device=DEV),
                      torch.ones(1, dtype=torch.int32, device=DEV), 0.1, workspace=small)
    with pytest.raises(ops.PagedKVError):
        ops.pa_decode(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, float("nan"))


def test_write_and_copy_bit_exact_all_dtypes(ops):
    for dtype in (torch.float32, torch.float16, torch.bfloat16):
        g = torch.Generator().manual_seed(11)
        NB, Hkv, B, D, T = 40, 3, 8, 64, 25
        kc = W.randn((NB, Hkv, B, D), dtype, g)
        vc = W.randn((NB, Hkv, B, D), dtype, g)
        key = W.randn((T, Hkv, D), dtype, g)
        val = W.randn((T, Hkv, D), dtype, g)
        slots = torch.randperm(NB * B, generator=g)[:T].to(torch.int64)
        slots[3] = -1
        pairs = torch.tensor([[1, 30], [2, 31], [5, 39]], dtype=torch.int64)
        kg, vg = kc.to(DEV), vc.to(DEV)
        err = ops.new_error_word(DEV)
        ops.pa_copy_blocks(kg, vg, pairs.to(DEV), err=err)
        ops.pa_write_kv(key.to(DEV), val.to(DEV), kg, vg, slots.to(DEV), err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        native.copy_blocks(kc, vc, pairs.numpy())
        native.write_kv(key, val, kc, vc, slots.numpy())
        assert torch.equal(kg.cpu(), kc) and torch.equal(vg.cpu(), vc)
