"""The kernels' bounded waits end a call that would otherwise wait forever.

Every mbarrier wait in the decode counts SM cycles and gives up after a
limit: it sets PA_DEVERR_TIMEOUT, tells the CTA's other warps to stop (the
producer issues nothing more and waits for its own copies in flight), and the
kernel returns, so the context stays usable (cf-1.com news/5879632, section
6.3, on waits that never end).  A test build of the library (build variant
``faulttest``) makes one wait run out without any fault: its producer never
issues the first ring entry of the CTA that owns the step's first tile -- no
copy, no arrival -- and its wait limit is 1e9 cycles (about half a second).  The call must come back with the TIMEOUT
bit set; a following normal call on a freshly zeroed workspace must match the
oracle.  Nothing here traps, faults or hangs the GPU.
"""
import time

import pytest
import torch

from gpu_utils import assert_attention_close
from oracle import native
from paged_kv_cache_170_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_170_gb300 import build

    build.build()
    path = build.build(variant="faulttest")
    from paged_kv_cache_170_gb300 import ops

    return ops, ops._load(path)


def _call_decode(ops, lib, inp, out, workspace, err):
    NB, Hkv, B, D = inp.k_cache.shape
    S, Hq, _ = inp.q.shape
    return lib.pa_decode(out.data_ptr(), inp.q.data_ptr(), inp.k_cache.data_ptr(), inp.v_cache.data_ptr(),
                         inp.block_tables.data_ptr(), inp.block_tables.shape[1], inp.context_lens.data_ptr(), S, Hq,
                         Hkv, D, B, NB, float(inp.scale), ops._DTYPES[inp.q.dtype], workspace.data_ptr(),
                         workspace.numel(), err.data_ptr(), torch.cuda.current_stream().cuda_stream)


CASES = {
    # tensor-core kernel (bf16, B = 16) and CUDA-core kernel (fp32)
    "gqa_bf16": lambda: W.make_inputs(W.scaled(W.GQA, num_seqs=6, num_blocks=6 * 256 + 5, ctx_min=500), 3),
    "tiny_f32": lambda: W.make_inputs(W.TINY, 0),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_a_wait_that_runs_out_sets_timeout_and_returns(libs, case):
    ops, flib = libs
    cpu = CASES[case]()
    inp = cpu.to(DEV)
    S, Hq, D = inp.q.shape
    Hkv = inp.k_cache.shape[1]
    ws = ops.new_workspace(S, Hq, Hkv, D, DEV)
    err = ops.new_error_word(DEV)
    out = torch.zeros_like(inp.q)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert _call_decode(ops, flib, inp, out, ws, err) == 0
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert "TIMEOUT" in ops.error_names(int(err.item()))
    assert elapsed < 20.0, elapsed  # a few wait limits at most, never an endless wait

    # the context is still usable, and a normal call on a fresh workspace is right
    ws2 = ops.new_workspace(S, Hq, Hkv, D, DEV)
    err2 = ops.new_error_word(DEV)
    out2 = torch.full_like(inp.q, float("nan"))
    assert _call_decode(ops, ops.lib, inp, out2, ws2, err2) == 0
    torch.cuda.synchronize()
    assert int(err2.item()) == 0, ops.error_names(int(err2.item()))
    ref = native.decode(cpu.q, cpu.k_cache, cpu.v_cache, cpu.block_tables.numpy(), cpu.context_lens.numpy(),
                        cpu.scale)
    assert_attention_close(out2, ref, strict=cpu.q.dtype != torch.float32)
