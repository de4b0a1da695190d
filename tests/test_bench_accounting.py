"""The benchmark's byte accounting (host only): the logical, distinct and
algorithmic bytes of a decode step that its roofline divides by time, counted
here by hand on small workloads."""
import torch

import bench
from paged_kv_cache_170_gb300 import scenarios
from paged_kv_cache_170_gb300 import workloads as W


def _prefix_small():
    return scenarios.shared_prefix_inputs(0, num_parents=4, prefix_tokens=256, suffix_max=300,
                                          w=W.scaled(W.PREFIX, num_blocks=300, max_blocks_per_seq=40))


def test_logical_and_algorithmic_bytes_of_the_tiny_workload():
    inp = W.make_inputs(W.TINY, 0)  # fp32, lengths 10, 3, 16, 1; 2 kv heads of 64; B = 4
    row = 2 * 64 * 4  # K + V bytes of one token of one kv head
    assert bench.kv_bytes(inp) == (10 + 3 + 16 + 1) * 2 * row
    entries = (3 + 1 + 4 + 1) * 2  # table entries read: blocks per sequence, per kv head
    q_out = 2 * 4 * 2 * 64 * 4
    assert bench.algorithmic_bytes(inp) == bench.kv_bytes(inp) + q_out + entries * 4 + 4 * 4
    # pa_write_decode adds its write: the new rows read and stored, a table entry and a length per sequence
    new_rows = 2 * 2 * (4 * 2 * 64 * 4)
    assert bench.algorithmic_bytes(inp, with_write=True) == bench.algorithmic_bytes(inp) + new_rows + 8 * 4


def test_distinct_bytes_count_a_shared_block_once():
    inp = W.make_inputs(W.TINY, 0)
    assert bench.unique_kv_bytes(inp) == bench.kv_bytes(inp)  # nothing shared
    shared = _prefix_small()
    B, Hkv, D = shared.k_cache.shape[2], shared.k_cache.shape[1], shared.k_cache.shape[3]
    per_token = Hkv * D * shared.k_cache.element_size() * 2
    # by hand: every physical block once, with the most valid rows any sharer reads from it
    rows = {}
    for s in range(shared.q.shape[0]):
        L = int(shared.context_lens[s])
        for b in range((L + B - 1) // B):
            pid = int(shared.block_tables[s, b])
            rows[pid] = max(rows.get(pid, 0), min(B, L - b * B))
    assert bench.unique_kv_bytes(shared) == sum(rows.values()) * per_token
    assert bench.unique_kv_bytes(shared) < bench.kv_bytes(shared)


def test_l2_flush_policy_and_kernel_names():
    assert not bench.needs_l2_flush(W.make_inputs(W.TINY, 0), "warm")
    assert bench.needs_l2_flush(W.make_inputs(W.TINY, 0), "auto")  # 30 KB of K/V would sit in L2
    tiny = W.make_inputs(W.TINY, 0)
    assert bench.decode_kernel_name(tiny, shared=False) == "decode_partition_kernel"  # fp32: CUDA cores
    gqa_like = W.make_inputs(W.scaled(W.GQA, num_seqs=2, num_blocks=2 * 256 + 3), 0)
    assert bench.decode_kernel_name(gqa_like, shared=False) == "decode_partition_mma_kernel"
    assert bench.decode_kernel_name(gqa_like, shared=False, fused=True).startswith("append_last_kernel + ")


def test_flush_writes_then_reads_its_buffer():
    buf = torch.zeros(1 << 12, dtype=torch.uint8)
    bench.flush_l2(buf, 300)
    assert int(buf[0]) == 300 & 255 and bool((buf == buf[0]).all())


def test_profile_hash_ignores_trace_blocks_but_not_their_else_branch():
    src = ["int a;", "#ifdef PA_TRACE", "#if X", "t();", "#endif", "u();", "#endif", "int b;",
           "#ifdef PA_TRACE", "v();", "#else", "w();", "#endif", "  ", "int c;"]
    assert bench._product_lines(src) == ["int a;", "int b;", "#ifndef PA_TRACE", "w();", "#endif", "int c;"]
    # a product line inside a trace block's else branch is part of the hash
    assert bench._product_lines(src[:11] + ["x();"] + src[12:]) != bench._product_lines(src)
    assert bench._product_lines(["#ifdef PA_TRACE", "z();", "#endif"]) == []
