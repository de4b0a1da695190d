"""Host logic of the decode step (no GPU): when a step can run its write and
decode as one pa_write_decode call."""
import torch

from paged_kv_cache_170_gb300 import scenarios, step
from paged_kv_cache_170_gb300 import workloads as W


def test_plain_workloads_append_one_token_per_sequence():
    assert step.one_token_per_sequence(W.make_inputs(W.TINY, 0))
    inp = scenarios.shared_prefix_inputs(0, num_parents=4, prefix_tokens=256, suffix_max=300,
                                         w=W.scaled(W.PREFIX, num_blocks=300, max_blocks_per_seq=40))
    assert inp.copy_pairs.numel() > 0  # copy-on-write copies still run first, as their own kernel
    assert step.one_token_per_sequence(inp)


def test_other_token_layouts_keep_the_separate_write():
    inp = W.make_inputs(W.TINY, 0)
    moved = inp.to("cpu")
    moved.new_pos = moved.new_pos.clone()
    moved.new_pos[1] -= 1  # not the sequence's last position
    assert not step.one_token_per_sequence(moved)
    fewer = inp.to("cpu")
    fewer.new_seq, fewer.new_pos = fewer.new_seq[:2], fewer.new_pos[:2]  # not every sequence appends
    assert not step.one_token_per_sequence(fewer)
    empty = inp.to("cpu")
    empty.context_lens = empty.context_lens.clone()
    empty.context_lens[3] = 0  # an empty sequence has no position to write
    empty.new_pos = (empty.context_lens.to(torch.int64) - 1).to(torch.int32)
    assert not step.one_token_per_sequence(empty)
