"""pa_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers have no device allocator of their own, must not call cudaMalloc
on their path (it can synchronise the whole device), or run where all device
memory is already reserved.  For them the library keeps the decode scratch in
a static 4 MiB device array.  This checks, through the C ABI, that the call
gives the same output as pa_decode with a caller workspace, twice in a row on
different inputs (the array keeps the previous call's contents), and that a
shape needing more scratch than the array holds is refused.

Kept in a file of its own, collected after every other test file.
"""
import pytest
import torch

from gpu_utils import assert_attention_close
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


def _case(seed, num_seqs, ctx_min, ctx_max):
    w = W.scaled(W.GQA, num_seqs=num_seqs, num_blocks=num_seqs * 256 + 7, ctx_min=ctx_min, ctx_max=ctx_max)
    return W.make_inputs(w, seed).to("cuda")


def test_noalloc_matches_workspace_decode_on_two_calls(ops):
    for call, (seed, S, lo, hi) in enumerate([(1, 6, 1, 4096), (2, 9, 300, 2000)]):
        inp = _case(seed, S, lo, hi)
        err = ops.new_error_word("cuda")
        ref = ops.pa_decode(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale,
                            err=err)
        out = torch.full_like(inp.q, float("nan"))
        ops.pa_decode_noalloc(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale,
                              out=out, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, ops.error_names(int(err.item()))
        assert_attention_close(out, ref.double().cpu().numpy(), strict=False)


def test_noalloc_refuses_shapes_beyond_its_scratch(ops):
    S = 300_000  # needs more than 4 MiB of scratch; refused before any device work
    need = ops.pa_decode_workspace_size(S, 32, 8, 128)
    assert need > 4 << 20
    dummy = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    status = ops.lib.pa_decode_noalloc(dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(),
                                       dummy.data_ptr(), 1, dummy.data_ptr(), S, 32, 8, 128, 16, 1, 0.1, 2, None,
                                       None)
    assert ops.lib.pa_status_string(status) == b"PA_ERR_WORKSPACE"
