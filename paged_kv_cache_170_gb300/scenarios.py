"""The two sharing workloads, built by replaying block-manager operations.

* shared prefix: parents fork a common prompt, grow private suffixes that end
  in a partly filled block, and are forked once more; every sequence then
  appends one token, so the first of each pair writes into a tail block with
  count 2 and triggers a copy-on-write (aiqz.cc "paged-attention-mechanism",
  section "前缀共享机制"; cf-1.com news/5879632, section 4.2).
* long-context parallel sampling: n branches fork one long prompt (best-of-n /
  beam style sharing, cf-1.com news/5879632, section 4.1) and grow suffixes.

Random draws come from ``workloads``; the block tables, slots and copy pairs
come from the host ``BlockManager``.
"""
from __future__ import annotations

import torch

from .block_manager import BlockManager
from .workloads import (DecodeInputs, LONGCTX, PREFIX, Workload, cpu_generator, draw_pools, randn,
                        scaled)


def _finish(w: Workload, mgr: BlockManager, seqs: list, gen, device, seed, extra) -> DecodeInputs:
    """Every sequence appends one token (the step's write), then the inputs are collected."""
    slots, pairs = [], []
    for s in seqs:
        slot, cow = mgr.append_slot(s)
        slots.append(slot)
        if cow is not None:
            pairs.append(cow)
    mgr.check()
    tables = torch.from_numpy(mgr.block_tables(seqs, width=w.max_blocks_per_seq))
    lens = torch.from_numpy(mgr.context_lens(seqs))
    S, Hq, Hkv, D = len(seqs), w.num_heads, w.num_kv_heads, w.head_dim
    q = randn((S, Hq, D), w.dtype, gen)
    new_key = randn((S, Hkv, D), w.dtype, gen)
    new_value = randn((S, Hkv, D), w.dtype, gen)
    k_cache, v_cache = draw_pools(w, gen, device, seed)
    extra = dict(extra)
    extra.update(manager_slots=torch.tensor(slots, dtype=torch.int64),
                 unique_blocks=mgr.num_used_blocks(), manager=mgr)
    inp = DecodeInputs(w, q, k_cache, v_cache, tables, lens, new_key, new_value,
                       torch.arange(S, dtype=torch.int32), (lens.to(torch.int64) - 1).to(torch.int32),
                       torch.tensor(pairs, dtype=torch.int64).reshape(-1, 2), float(D) ** -0.5, extra)
    return inp.to(device)


def shared_prefix_inputs(seed: int = 0, device="cpu", num_parents: int = 64, prefix_tokens: int = 1024,
                         suffix_max: int = 1024, w: Workload = PREFIX) -> DecodeInputs:
    gen = cpu_generator(seed)
    w = scaled(w, num_seqs=2 * num_parents)
    mgr = BlockManager(w.num_blocks, w.block_size, torch.randperm(w.num_blocks, generator=gen).tolist())
    mgr.allocate("prompt", prefix_tokens)
    seqs = []
    suffixes = []
    for i in range(num_parents):
        while True:  # the parents' last block must be partly filled
            s = int(torch.randint(w.ctx_min, suffix_max + 1, (1,), generator=gen))
            if s % w.block_size:
                break
        suffixes.append(s)
        mgr.fork(("p", i), "prompt")
        for _ in range(s):
            mgr.append_slot(("p", i))
        mgr.fork(("c", i), ("p", i))
        seqs += [("p", i), ("c", i)]
    mgr.free_seq("prompt")
    return _finish(w, mgr, seqs, gen, device, seed, dict(suffixes=suffixes, prefix_tokens=prefix_tokens))


def long_context_inputs(seed: int = 0, device="cpu", num_prompts: int = 8, branches: int = 4,
                        prompt_tokens: int = 32768, suffix_max: int = 512,
                        w: Workload = LONGCTX) -> DecodeInputs:
    gen = cpu_generator(seed)
    w = scaled(w, num_seqs=num_prompts * branches)
    mgr = BlockManager(w.num_blocks, w.block_size, torch.randperm(w.num_blocks, generator=gen).tolist())
    seqs, suffixes = [], []
    for i in range(num_prompts):
        mgr.allocate(("prompt", i), prompt_tokens)
        for j in range(branches):
            s = int(torch.randint(w.ctx_min, suffix_max + 1, (1,), generator=gen))
            suffixes.append(s)
            mgr.fork(("b", i, j), ("prompt", i))
            for _ in range(s - 1):      # the last suffix token is the step's write
                mgr.append_slot(("b", i, j))
            seqs.append(("b", i, j))
        mgr.free_seq(("prompt", i))
    return _finish(w, mgr, seqs, gen, device, seed, dict(suffixes=suffixes, prompt_tokens=prompt_tokens))
