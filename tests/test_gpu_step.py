"""The decode step recorded as CUDA graphs (paged_kv_cache_170_gb300.step):
replays give the oracle's result and exactly what kernel-by-kernel launches
give, and follow inputs that the caller updates in place between replays."""
import pytest
import torch

from gpu_utils import assert_attention_close, oracle_step
from paged_kv_cache_170_gb300 import scenarios
from paged_kv_cache_170_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def step_mod():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_170_gb300 import build

    build.build()
    from paged_kv_cache_170_gb300 import step

    return step


def _case(name, seed=0):
    if name == "gqa":
        return W.make_inputs(W.scaled(W.GQA, num_seqs=5, num_blocks=5 * 256 + 9), seed)
    if name == "mha":
        return W.make_inputs(W.scaled(W.MHA, num_seqs=7, num_blocks=1000), seed)
    if name == "prefix":  # has copy-on-write pairs
        return scenarios.shared_prefix_inputs(seed, num_parents=4, prefix_tokens=256, suffix_max=300,
                                              w=W.scaled(W.PREFIX, num_blocks=300, max_blocks_per_seq=40))
    raise KeyError(name)


@pytest.mark.parametrize("name", ["gqa", "mha", "prefix"])
def test_graph_step_matches_oracle_and_eager(step_mod, name):
    inp_cpu = _case(name)
    _, kc, vc, ref = oracle_step(inp_cpu)

    eager_in = inp_cpu.to("cuda")
    eager = step_mod.DecodeStep(eager_in, graphs=False)
    out_e = eager.run().clone()

    graph_in = inp_cpu.to("cuda")
    runner = step_mod.DecodeStep(graph_in, graphs=True)
    for _ in range(3):  # replays repeat the same step (the copies and writes are idempotent)
        out_g = runner.run()
    torch.cuda.synchronize()
    assert int(runner.err.item()) == 0 and int(eager.err.item()) == 0
    assert torch.equal(out_g, out_e)
    assert torch.equal(graph_in.k_cache.cpu(), kc) and torch.equal(graph_in.v_cache.cpu(), vc)
    assert_attention_close(out_g, ref, strict=False)


def test_graph_step_follows_inputs_updated_in_place(step_mod):
    inp_cpu = _case("gqa", seed=3)
    dev_in = inp_cpu.to("cuda")
    runner = step_mod.DecodeStep(dev_in, graphs=True)
    from paged_kv_cache_170_gb300 import ops

    g = torch.Generator(device="cpu").manual_seed(11)
    for _ in range(2):
        # a new step: new queries and new token rows, written into the captured buffers
        dev_in.q.copy_(torch.randn(dev_in.q.shape, generator=g).to(dev_in.q.dtype))
        dev_in.new_key.copy_(torch.randn(dev_in.new_key.shape, generator=g).to(dev_in.new_key.dtype))
        dev_in.new_value.copy_(torch.randn(dev_in.new_value.shape, generator=g).to(dev_in.new_value.dtype))
        out_g = runner.run().clone()
        ref = ops.pa_decode(dev_in.q, dev_in.k_cache, dev_in.v_cache, dev_in.block_tables, dev_in.context_lens,
                            dev_in.scale)
        torch.cuda.synchronize()
        assert int(runner.err.item()) == 0
        assert torch.equal(out_g, ref)
        _, _, _, oref = oracle_step(dev_in.to("cpu"))
        assert_attention_close(out_g, oref, strict=False)


@pytest.mark.parametrize("name", ["prefix"])
def test_graph_step_with_shared_decode(step_mod, name):
    inp_cpu = _case(name)
    _, _, _, ref = oracle_step(inp_cpu)
    runner = step_mod.DecodeStep(inp_cpu.to("cuda"), graphs=True, shared=True)
    assert runner.plan_info["num_groups"] > 0
    for _ in range(2):
        out = runner.run()
    torch.cuda.synchronize()
    assert int(runner.err.item()) == 0
    assert_attention_close(out, ref, strict=True)


def test_step_pipeline_outputs_follow_host_inputs(step_mod):
    """StepPipeline: new queries written into each step's host buffer (after
    that slot's previous upload) come back, step by step, as exactly what
    pa_decode gives on them."""
    from paged_kv_cache_170_gb300 import ops

    inp_cpu = _case("gqa", seed=5)
    dev_in = inp_cpu.to("cuda")
    pipe = step_mod.StepPipeline(dev_in, graphs=True)
    g = torch.Generator(device="cpu").manual_seed(12)
    qs, outs, pending = [], [], None
    for k in range(6):
        sl = pipe.slots[k % 2]
        sl.ev_up.synchronize()  # the slot's previous upload has read its host buffer
        q = torch.randn(dev_in.q.shape, generator=g).to(dev_in.q.dtype)
        sl.packed.host_views["q"].copy_(q)
        qs.append(q)
        pipe.step()
        if pending is not None:  # the previous step's output, read before its slot is reused
            pending.ev_down.synchronize()
            outs.append(pending.out_host.clone())
        pending = sl
    pending.ev_down.synchronize()
    outs.append(pending.out_host.clone())
    torch.cuda.synchronize()
    for sl in pipe.slots:
        assert int(sl.runner.err.item()) == 0
    for q, out in zip(qs, outs):
        ref = ops.pa_decode(q.to("cuda"), dev_in.k_cache, dev_in.v_cache, dev_in.block_tables, dev_in.context_lens,
                            dev_in.scale)
        torch.cuda.synchronize()
        assert torch.equal(out, ref.cpu())
