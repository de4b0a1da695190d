"""pa_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers have no device allocator of their own, must not call cudaMalloc
on their path (it can synchronise the whole device), or run where all device
memory is already reserved.  For them the library keeps the decode scratch in
a static 4 MiB device array.  This checks, through the C ABI, that calls in a
row on different shapes and dtypes (a larger shape between the smaller ones,
so that anything a call left in the shared array would show) give exactly
pa_decode's output with a caller workspace: same kernel, same grid, same
inputs, so the outputs must be bit-identical.  It also checks that a shape
needing more scratch than the array holds is refused.

Kept in a file of its own, collected after every other test file.
"""
import pytest
import torch

from gpu_utils import assert_attention_close
from oracle import native
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


def _gqa(seed, num_seqs, ctx_min, ctx_max):
    return W.make_inputs(W.scaled(W.GQA, num_seqs=num_seqs, num_blocks=num_seqs * 256 + 7, ctx_min=ctx_min,
                                  ctx_max=ctx_max), seed, device="cuda")


# (name, cpu inputs): bf16 GQA and f16 MHA take the tensor-core kernel, the
# fp32 tiny case the CUDA-core one; the large GQA call sits between the
# smaller checked ones
CALLS = [
    ("gqa_bf16_small", lambda: _gqa(1, 6, 1, 4096)),
    ("gqa_bf16_large", lambda: _gqa(3, 40, 2000, 4096)),
    ("gqa_bf16_small_again", lambda: _gqa(2, 9, 300, 2000)),
    ("mha_f16", lambda: W.make_inputs(W.scaled(W.MHA, num_seqs=5, num_blocks=700), 4, device="cuda")),
    ("tiny_f32", lambda: W.make_inputs(W.TINY, 0, device="cuda")),
]


def test_noalloc_matches_workspace_decode_on_calls_in_a_row(ops):
    for name, make in CALLS:
        inp = make()
        err = ops.new_error_word("cuda")
        ref = ops.pa_decode(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale,
                            err=err)
        out = torch.full_like(inp.q, float("nan"))
        ops.pa_decode_noalloc(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale,
                              out=out, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, (name, ops.error_names(int(err.item())))
        assert torch.equal(out, ref), f"{name}: pa_decode_noalloc differs from pa_decode"
        if name == "tiny_f32":
            # and both agree with the oracle's decode of the same pools
            cpu = inp.to("cpu")
            out_ref = native.decode(cpu.q, cpu.k_cache, cpu.v_cache, cpu.block_tables.numpy(),
                                    cpu.context_lens.numpy(), cpu.scale)
            assert_attention_close(out, out_ref)


def test_noalloc_refuses_shapes_beyond_its_scratch(ops):
    S = 300_000  # needs more than 4 MiB of scratch; refused before any device work
    need = ops.pa_decode_workspace_size(S, 32, 8, 128)
    assert need > 4 << 20
    dummy = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    status = ops.lib.pa_decode_noalloc(dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(),
                                       dummy.data_ptr(), 1, dummy.data_ptr(), S, 32, 8, 128, 16, 1, 0.1, 2, None,
                                       None)
    assert ops.lib.pa_status_string(status) == b"PA_ERR_WORKSPACE"


def test_noalloc_refuses_bad_arguments_before_enqueueing(ops):
    dummy = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    p = dummy.data_ptr()
    # a null table pointer and a misaligned output are refused, as pa_decode refuses them
    assert ops.lib.pa_decode_noalloc(p, p, p, p, None, 1, p, 4, 32, 8, 128, 16, 1, 0.1, 2, None, None) == 1
    assert ops.lib.pa_decode_noalloc(p + 2, p, p, p, p, 1, p, 4, 32, 8, 128, 16, 1, 0.1, 2, None, None) == 1
    with pytest.raises(ValueError):
        # the binding checks shapes: an out smaller than q is refused before the call
        inp = _gqa(5, 2, 16, 64)
        ops.pa_decode_noalloc(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale,
                              out=torch.empty_like(inp.q)[:1])
