"""Parity of pa_write_decode (each sequence's new token written at position
context_len - 1, then decode attention, the decode launched while the write
runs) with the CPU oracle's write followed by its decode, through the C ABI.

The pools after the call must equal the oracle's pools bit for bit; the
output is held to the decode tolerances (fp16/bf16 max abs 2e-3 and max rel
1e-2 over |ref| >= 1e-2; fp32 abs 1e-5 + rel 1e-4) and must be bit-identical
to the separate write + pa_decode path, which reads the same tile contents.
"""
import numpy as np
import pytest
import torch

from gpu_utils import assert_attention_close, oracle_step
from oracle import native
from paged_kv_cache_170_gb300 import step as step_mod
from paged_kv_cache_170_gb300 import workloads as W
from test_gpu_parity import _full_case, random_case, small_case

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


def fused_step(ops, inp):
    """Copy-on-write copies (if any), then one pa_write_decode call."""
    assert step_mod.one_token_per_sequence(inp)
    err = ops.new_error_word(inp.q.device)
    if inp.copy_pairs.numel():
        ops.pa_copy_blocks(inp.k_cache, inp.v_cache, inp.copy_pairs, err)
    out = ops.pa_write_decode(inp.q, inp.new_key, inp.new_value, inp.k_cache, inp.v_cache, inp.block_tables,
                              inp.context_lens, inp.scale, err=err)
    torch.cuda.synchronize()
    return out, int(err.item())


@pytest.mark.parametrize("name", ["tiny", "mha_small", "gqa_small", "prefix_small", "longctx_small"])
def test_write_decode_small(ops, name):
    cpu = small_case(name)
    fused_in, split_in = cpu.to(DEV), cpu.to(DEV)
    out, err = fused_step(ops, fused_in)
    assert err == 0, ops.error_names(err)
    _, kc_ref, vc_ref, out_ref = oracle_step(cpu)
    assert torch.equal(fused_in.k_cache.cpu(), kc_ref) and torch.equal(fused_in.v_cache.cpu(), vc_ref)
    assert_attention_close(out, out_ref, strict=True)
    split = ops.decode_step(split_in)
    torch.cuda.synchronize()
    assert torch.equal(out, split)


def oracle_write_decode(q, kc, vc, tables, lens, new_key, new_value, scale):
    """The oracle's write of each sequence's token at position len - 1, then its decode."""
    kc, vc = kc.clone(), vc.clone()
    B = kc.shape[2]
    seqs = np.nonzero(lens.numpy() > 0)[0].astype(np.int32)
    pos = (lens.numpy()[seqs] - 1).astype(np.int32)
    slots = native.slot_mapping(tables.numpy(), seqs, pos, B)
    native.write_kv(new_key[torch.as_tensor(seqs, dtype=torch.long)], new_value[torch.as_tensor(seqs, dtype=torch.long)],
                    kc, vc, slots)
    return kc, vc, native.decode(q, kc, vc, tables.numpy(), lens.numpy(), scale)


CASES = {
    # name: (lens, Hq, Hkv, D, B, dtype, pad_tables)
    # empty sequences, tails of one token, full last blocks
    "zero_one_full_tails": ([0, 1, 0, 2, 16, 17, 32, 33], 8, 2, 128, 16, torch.bfloat16, True),
    # two head chunks per kv head (G = 16)
    "group16_two_chunks": ([300, 45, 1, 4096], 32, 2, 128, 32, torch.bfloat16, True),
    # long sequences cut among several CTAs next to short ones
    "cut_pairs": ([20000, 5, 9000, 16, 12345], 8, 8, 128, 16, torch.float16, True),
    "d64_b64": ([64, 65, 1, 700], 8, 4, 64, 64, torch.bfloat16, True),
    "gqa3_b48": ([47, 48, 49, 1000], 6, 2, 128, 48, torch.float16, False),
    # CUDA-core decode paths
    "fp32": ([3, 130, 64, 0, 9], 4, 2, 128, 8, torch.float32, True),
    "block8_bf16": ([7, 8, 9, 300], 8, 2, 64, 8, torch.bfloat16, True),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_write_decode_cases(ops, name):
    lens, Hq, Hkv, D, B, dtype, pad = CASES[name]
    q, kc, vc, tables, lens_t = random_case(lens, Hq, Hkv, D, B, dtype, seed=len(name) + 40, pad_tables=pad)
    g = torch.Generator().manual_seed(len(name))
    nk = W.randn((len(lens), Hkv, D), dtype, g)
    nv = W.randn((len(lens), Hkv, D), dtype, g)
    scale = D ** -0.5
    kg, vg = kc.to(DEV), vc.to(DEV)
    err = ops.new_error_word(DEV)
    out = ops.pa_write_decode(q.to(DEV), nk.to(DEV), nv.to(DEV), kg, vg, tables.to(DEV), lens_t.to(DEV), scale,
                              err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, ops.error_names(int(err.item()))
    kc_ref, vc_ref, ref = oracle_write_decode(q, kc, vc, tables, lens_t, nk, nv, scale)
    assert torch.equal(kg.cpu(), kc_ref) and torch.equal(vg.cpu(), vc_ref)
    assert_attention_close(out, ref, strict=False)
    for s, L in enumerate(lens):
        if L == 0:
            assert torch.count_nonzero(out[s]) == 0
    # the same result as the separate write, then pa_decode
    again = ops.pa_decode(q.to(DEV), kg, vg, tables.to(DEV), lens_t.to(DEV), scale)
    assert torch.equal(out, again)


@pytest.mark.parametrize("name,sample", [("gqa", None), ("mha", None), ("prefix", None),
                                         ("longctx", [0, 5, 10, 15, 21, 31])])
def test_write_decode_full_size(ops, name, sample):
    """The full-size workloads as the benchmark's default step runs them
    (copy-on-write copies, then pa_write_decode); the oracle checks every
    sequence (or the listed sample)."""
    inp = _full_case(name)
    cpu = inp.to("cpu")
    out, err = fused_step(ops, inp)
    assert err == 0, ops.error_names(err)
    _, kc_ref, vc_ref, out_ref = oracle_step(cpu, seqs=sample)
    assert torch.equal(inp.k_cache.cpu(), kc_ref) and torch.equal(inp.v_cache.cpu(), vc_ref)
    got = out if sample is None else out[torch.as_tensor(sample, device=out.device)]
    print(name, assert_attention_close(got, out_ref, strict=True))


def test_fused_step_graphs_match_eager_and_oracle(ops):
    cpu = small_case("gqa_small", seed=5)
    eager_in, graph_in = cpu.to(DEV), cpu.to(DEV)
    eager = step_mod.DecodeStep(eager_in, graphs=False)
    assert eager.fused and eager.launches_per_step == 2 and not eager.has_pre
    a = eager.run().clone()
    runner = step_mod.DecodeStep(graph_in, graphs=True)
    for _ in range(3):
        b = runner.run()
    torch.cuda.synchronize()
    assert int(runner.err.item()) == 0
    assert torch.equal(a, b)
    _, kc_ref, vc_ref, out_ref = oracle_step(cpu)
    assert torch.equal(graph_in.k_cache.cpu(), kc_ref) and torch.equal(graph_in.v_cache.cpu(), vc_ref)
    assert_attention_close(b, out_ref, strict=True)


def test_write_decode_bad_block_id_sets_error_bit(ops):
    q, kc, vc, tables, lens = random_case([40, 20], 4, 2, 128, 16, torch.bfloat16, seed=5, pad_tables=True)
    NB = kc.shape[0]
    bad = tables.clone()
    bad[1, 1] = NB + 7  # the block that holds sequence 1's new token (position 19)
    nk = torch.zeros(2, 2, 128, dtype=torch.bfloat16, device=DEV)
    kg, vg = kc.to(DEV), vc.to(DEV)
    err = ops.new_error_word(DEV)
    ops.pa_write_decode(q.to(DEV), nk, nk, kg, vg, bad.to(DEV), lens.to(DEV), 0.1, err=err)
    torch.cuda.synchronize()
    assert "BLOCK_ID" in ops.error_names(int(err.item()))
    # sequence 0's token (position 39: block 2, offset 7) was written; nothing else changed
    kc[tables[0, 2], :, 7] = 0
    vc[tables[0, 2], :, 7] = 0
    assert torch.equal(kg.cpu(), kc) and torch.equal(vg.cpu(), vc)


def test_write_decode_host_validation(ops):
    inp = small_case("gqa_small").to(DEV)
    with pytest.raises(ValueError):
        ops.pa_write_decode(inp.q, inp.new_key[:1], inp.new_value[:1], inp.k_cache, inp.v_cache, inp.block_tables,
                            inp.context_lens, inp.scale)
