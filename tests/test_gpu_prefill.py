"""pa_prefill (prompt attention through the block table) against the float64
oracle: ragged prompts with and without cached history, one-token prompts,
empty prompts, partly filled last blocks, head groups of 1, 4 and 8, head
dims 64 and 128, block sizes 16, 32 and 64, fp16 and bf16; the full-size prompt
workloads on sampled sequences; invariance under block relabelling."""
import math

import numpy as np
import pytest
import torch

from gpu_utils import assert_attention_close
from oracle import native
from paged_kv_cache_170_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def assert_prefill_close(got, ref):
    """The attention bar for a bf16 / fp16 output: max relative error <= 1e-2
    over |ref| >= 1e-2, and max absolute error <= 2e-3 where |ref| < 0.5.  A
    prompt's early rows see few tokens, so their outputs reach |out| ~ 1..4,
    where the rounding of the output alone (up to 2^-8 relative in bf16)
    exceeds 2e-3 absolute; below 0.5 half an ulp is under 1e-3."""
    stats = assert_attention_close(got, ref, strict=False)
    g = got.detach().float().cpu().double().numpy()
    err = np.abs(g - ref)
    big = np.abs(ref) >= 1e-2
    small = np.abs(ref) < 0.5
    max_rel = float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0
    max_abs_small = float(err[small].max()) if small.any() else 0.0
    assert max_rel <= 1e-2 and max_abs_small <= 2e-3, (max_rel, max_abs_small)
    return stats


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_170_gb300 import build

    build.build()
    from paged_kv_cache_170_gb300 import ops as _ops

    return _ops


def _case(lens, prompts, Hq, Hkv, D, B, dtype, seed=0, extra_blocks=7):
    g = torch.Generator().manual_seed(seed)
    S = len(lens)
    width = max(1, max(-(-L // B) for L in lens))
    NB = S * width + extra_blocks
    tables = torch.randperm(NB, generator=g)[:S * width].view(S, width).to(torch.int32)
    q_start = torch.zeros(S + 1, dtype=torch.int32)
    q_start[1:] = torch.cumsum(torch.tensor(prompts), 0).to(torch.int32)
    T = int(q_start[-1])
    q = torch.randn(T, Hq, D, generator=g).to(dtype)
    k = torch.randn(NB, Hkv, B, D, generator=g).to(dtype)
    v = torch.randn(NB, Hkv, B, D, generator=g).to(dtype)
    return q, k, v, tables, torch.tensor(lens, dtype=torch.int32), q_start


def _run(ops, q, k, v, tables, lens, q_start, scale):
    err = ops.new_error_word(DEV)
    args = [x.to(DEV) for x in (q, k, v, tables, lens, q_start)]
    n = (q_start[1:] - q_start[:-1]).max().item() if len(lens) else 0
    out = ops.pa_prefill(*args[:5], args[5], int(n), scale, err=err)
    torch.cuda.synchronize()
    return out, int(err.item())


CASES = {
    # name: (context lengths, prompt lengths, Hq, Hkv, D, B)
    "gqa_history": ([300, 129, 64, 17], [40, 129, 1, 17], 32, 8, 128, 16),
    "mha_ragged": ([97, 250, 33], [97, 80, 5], 4, 4, 128, 16),
    "g8_b32_d64": ([513, 40, 1], [200, 40, 1], 16, 2, 64, 32),
    "long_prompt": ([700], [700], 8, 2, 128, 16),
    "empty_prompts": ([50, 0, 80], [0, 0, 30], 8, 4, 64, 16),
    "b64_partial_last_block": ([200, 64, 130], [130, 64, 3], 8, 8, 128, 64),
    "g1_many_tiles": ([1100], [1000], 2, 2, 64, 16),
}


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_matches_oracle(ops, name, dtype):
    lens, prompts, Hq, Hkv, D, B = CASES[name]
    q, k, v, tables, L, qs = _case(lens, prompts, Hq, Hkv, D, B, dtype, seed=len(name))
    scale = 1.0 / math.sqrt(D)
    out, err = _run(ops, q, k, v, tables, L, qs, scale)
    assert err == 0, ops.error_names(err)
    ref = native.prefill(q, k, v, tables.numpy(), L.numpy(), qs.numpy(), scale)
    assert_prefill_close(out, ref)


@pytest.mark.parametrize("scale", [-0.07, 0.0])
def test_prefill_negative_and_zero_scale(ops, scale):
    lens, prompts = [300, 90], [200, 90]
    q, k, v, tables, L, qs = _case(lens, prompts, 8, 2, 128, 16, torch.bfloat16, seed=11)
    out, err = _run(ops, q, k, v, tables, L, qs, scale)
    assert err == 0, ops.error_names(err)
    assert_prefill_close(out, native.prefill(q, k, v, tables.numpy(), L.numpy(), qs.numpy(), scale))


def test_prefill_invariant_under_block_relabelling_and_deterministic(ops):
    lens, prompts = [300, 129], [100, 129]
    q, k, v, tables, L, qs = _case(lens, prompts, 16, 4, 128, 16, torch.bfloat16, seed=5)
    a, e1 = _run(ops, q, k, v, tables, L, qs, 0.1)
    NB = k.shape[0]
    pi = torch.randperm(NB, generator=torch.Generator().manual_seed(6))
    k2, v2 = torch.empty_like(k), torch.empty_like(v)
    k2[pi], v2[pi] = k, v
    b, e2 = _run(ops, q, k2, v2, pi[tables.long()].to(torch.int32), L, qs, 0.1)
    c, e3 = _run(ops, q, k, v, tables, L, qs, 0.1)
    assert e1 == e2 == e3 == 0
    assert torch.equal(a, b) and torch.equal(a, c)


@pytest.mark.parametrize("name,sample", [("prefill", [0, 5]), ("prefill_hist", [2, 7])])
def test_prefill_full_size_sampled(ops, name, sample):
    inp = W.make_prefill_inputs(W.WORKLOADS[name], 0, device=DEV)
    err = ops.new_error_word(DEV)
    out = ops.pa_prefill(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.q_start,
                         inp.max_q_len, inp.scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    cpu = inp.to("cpu")
    qs = cpu.q_start.numpy()
    for s in sample:
        # the oracle on this sequence alone (its rows, every 64th position and the last)
        rows = np.unique(np.r_[np.arange(qs[s], qs[s + 1], 64), qs[s + 1] - 1])
        sub_q = cpu.q[torch.as_tensor(rows, dtype=torch.long)]
        L = int(cpu.context_lens[s])
        n = int(qs[s + 1] - qs[s])
        # each chosen row is a one-row prompt of the context cut after its position
        for j, r in enumerate(rows):
            p = L - n + int(r - qs[s])
            ref = native.decode(sub_q[j:j + 1], cpu.k_cache, cpu.v_cache, cpu.block_tables.numpy()[s:s + 1],
                                np.array([p + 1], np.int32), cpu.scale)
            assert_prefill_close(out[int(r):int(r) + 1], ref)


def test_prefill_rejects_fp32_and_reports_overlong_prompts(ops):
    q, k, v, tables, L, qs = _case([40], [10], 4, 2, 64, 16, torch.float32)
    with pytest.raises(ops.PagedKVError, match="UNSUPPORTED"):
        _run(ops, q, k, v, tables, L, qs, 0.1)
    q, k, v, tables, L, qs = _case([100], [10], 4, 2, 64, 48, torch.bfloat16)  # 48 does not divide 64
    with pytest.raises(ops.PagedKVError, match="UNSUPPORTED"):
        _run(ops, q, k, v, tables, L, qs, 0.1)
    q, k, v, tables, L, qs = _case([40, 30], [10, 5], 4, 2, 64, 16, torch.bfloat16)
    L[1] = 3  # a prompt of 5 tokens in a context of 3
    out, err = _run(ops, q, k, v, tables, L, qs, 0.1)
    assert "CONTEXT" in ops.error_names(err)
