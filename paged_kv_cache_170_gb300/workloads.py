"""Seeded synthetic inputs for the paged decode workloads.

This module only draws numbers: context lengths, physical placements and
tensor values.  It holds none of the paged-attention arithmetic (no block
counts, no address computation, no attention): block-table rows are filled to
their full width with distinct physical ids, so no row length depends on a
context length.  The CUDA path and the oracle both consume what it returns.

Values are N(0, 1) rounded to the workload's dtype.  Small cases draw every
tensor from a CPU ``torch.Generator``; large pools are drawn on the device with
a CUDA generator seeded the same way (drawing a 1 GiB pool on host cores is
far too slow), and the oracle then checks sampled sequences copied back.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch


@dataclass(frozen=True)
class Workload:
    """Shape of one decode workload (one attention layer, one decode step)."""

    name: str
    num_seqs: int
    block_size: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: torch.dtype
    num_blocks: int            # physical blocks in each of the K and V pools
    max_blocks_per_seq: int    # block-table row width
    ctx_min: int               # context lengths drawn uniformly in [ctx_min, ctx_max]
    ctx_max: int
    fixed_lens: tuple = field(default=())   # explicit context lengths (overrides the draw)
    note: str = ""
    placement: str = "random"  # physical ids of a row: "random" permutation, or "contiguous" runs
    prompt_min: int = 0        # prefill workloads: prompt tokens per sequence drawn in [prompt_min, prompt_max]
    prompt_max: int = 0        # (the last positions of the context)


TINY = Workload("tiny", 4, 4, 2, 2, 64, torch.float32, 16, 4, 1, 16, fixed_lens=(10, 3, 16, 1),
                note="fp32 check; seq0 table [5, 1, 7]")
MHA = Workload("mha", 32, 16, 32, 32, 128, torch.float16, 6000, 128, 1, 2048,
               note="context lengths U[1, 2048] including the new token")
GQA = Workload("gqa", 64, 16, 32, 8, 128, torch.bfloat16, 20000, 256, 4096, 4096,
               note="Llama-3-8B-like layer, every context 4096")
# The two sharing workloads are built by replaying block-manager operations
# (see scenarios.py); these entries hold their shapes and draw ranges.
PREFIX = Workload("prefix", 128, 16, 32, 8, 128, torch.bfloat16, 8192, 128, 16, 1024,
                  note="64 parents x 2 forks; 1024-token shared prefix; suffix U[16, 1024], partial tail")
LONGCTX = Workload("longctx", 32, 32, 64, 8, 128, torch.bfloat16, 10000, 1040, 1, 512,
                   note="8 prompts x 4 branches; 32768-token prompt; branch suffix U[1, 512]")

# Prompt (prefill) steps of the GQA layer: the K/V of every context position,
# prompt included, already in the pools.
PREFILL = Workload("prefill", 8, 16, 32, 8, 128, torch.bfloat16, 1100, 128, 2048, 2048,
                   note="8 prompts of 2048 tokens, no history", prompt_min=2048, prompt_max=2048)
PREFILL_HIST = Workload("prefill_hist", 8, 16, 32, 8, 128, torch.bfloat16, 2100, 256, 4096, 4096,
                        note="8 sequences of 4096 tokens, the last 1024 are the prompt", prompt_min=1024,
                        prompt_max=1024)

WORKLOADS = {w.name: w for w in (TINY, MHA, GQA, PREFIX, LONGCTX, PREFILL, PREFILL_HIST)}


def scaled(w: Workload, **changes) -> Workload:
    """A smaller copy of a workload (for cases the oracle finishes in seconds)."""
    return replace(w, **changes)


def cpu_generator(seed: int) -> torch.Generator:
    return torch.Generator(device="cpu").manual_seed(seed)


def randn(shape, dtype: torch.dtype, gen: torch.Generator, device="cpu") -> torch.Tensor:
    """N(0, 1) drawn in float32 and rounded to ``dtype``."""
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(dtype)


def draw_lengths(w: Workload, gen: torch.Generator) -> torch.Tensor:
    if w.fixed_lens:
        return torch.tensor(w.fixed_lens, dtype=torch.int32)
    return torch.randint(w.ctx_min, w.ctx_max + 1, (w.num_seqs,), generator=gen, dtype=torch.int64).to(torch.int32)


def draw_full_tables(w: Workload, gen: torch.Generator) -> torch.Tensor:
    """Rows of ``max_blocks_per_seq`` distinct physical ids: from a random
    permutation of the pool, or (placement "contiguous") each row one run of
    consecutive ids, as an allocator that keeps a sequence's blocks together
    would give on a fresh pool."""
    need = w.num_seqs * w.max_blocks_per_seq
    if need > w.num_blocks:
        raise ValueError(f"{w.name}: {need} table entries do not fit a pool of {w.num_blocks}")
    if w.placement == "contiguous":
        ids = torch.arange(need)
    elif w.placement == "random":
        ids = torch.randperm(w.num_blocks, generator=gen)[:need]
    else:
        raise ValueError(f"unknown placement {w.placement!r}")
    return ids.view(w.num_seqs, w.max_blocks_per_seq).to(torch.int32).contiguous()


def draw_tiny_tables(gen: torch.Generator) -> torch.Tensor:
    """The 4 x 4 table of the fp32 check: seq0 is [5, 1, 7]; the other 13 ids are
    permuted and handed out in order (seq0 gets one more entry, then 4 each)."""
    rest = [i for i in range(16) if i not in (5, 1, 7)]
    order = torch.randperm(len(rest), generator=gen).tolist()
    ids = [rest[i] for i in order]
    rows = [[5, 1, 7, ids[0]], ids[1:5], ids[5:9], ids[9:13]]
    return torch.tensor(rows, dtype=torch.int32)


def draw_pools(w: Workload, gen_cpu: torch.Generator, device="cpu", seed: int = 0):
    """K and V pools [NB][Hkv][B][D], N(0, 1) in the workload dtype."""
    shape = (w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
    if torch.device(device).type == "cpu":
        return randn(shape, w.dtype, gen_cpu), randn(shape, w.dtype, gen_cpu)
    g = torch.Generator(device=device).manual_seed(seed + 7919)
    return randn(shape, w.dtype, g, device), randn(shape, w.dtype, g, device)


@dataclass
class DecodeInputs:
    """Everything one decode step consumes (pools already prefilled)."""

    workload: Workload
    q: torch.Tensor               # [S][Hq][D]
    k_cache: torch.Tensor         # [NB][Hkv][B][D]
    v_cache: torch.Tensor
    block_tables: torch.Tensor    # int32 [S][max_blocks]
    context_lens: torch.Tensor    # int32 [S]
    new_key: torch.Tensor         # [T][Hkv][D]
    new_value: torch.Tensor
    new_seq: torch.Tensor         # int32 [T]: sequence of new token i
    new_pos: torch.Tensor         # int32 [T]: its position in that sequence
    copy_pairs: torch.Tensor      # int64 [P][2] (src, dst); may be empty
    scale: float
    extra: dict = field(default_factory=dict)

    def to(self, device) -> "DecodeInputs":
        mv = lambda t: t.to(device) if isinstance(t, torch.Tensor) else t  # noqa: E731
        return DecodeInputs(self.workload, *(mv(getattr(self, n)) for n in (
            "q", "k_cache", "v_cache", "block_tables", "context_lens", "new_key", "new_value",
            "new_seq", "new_pos", "copy_pairs")), self.scale, dict(self.extra))


def make_inputs(w: Workload, seed: int = 0, device="cpu") -> DecodeInputs:
    """Inputs of the plain (unshared) workloads: tiny, mha, gqa and scaled copies.

    The step writes one new token per sequence, at position context_len - 1,
    then decodes over the whole context including it.
    """
    gen = cpu_generator(seed)
    lens = draw_lengths(w, gen)
    tables = draw_tiny_tables(gen) if w.name == "tiny" else draw_full_tables(w, gen)
    S, Hq, Hkv, D = w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim
    q = randn((S, Hq, D), w.dtype, gen)
    new_key = randn((S, Hkv, D), w.dtype, gen)
    new_value = randn((S, Hkv, D), w.dtype, gen)
    k_cache, v_cache = draw_pools(w, gen, device, seed)
    new_seq = torch.arange(S, dtype=torch.int32)
    new_pos = (lens.to(torch.int64) - 1).clamp(min=0).to(torch.int32)
    keep = lens > 0
    inp = DecodeInputs(w, q, k_cache, v_cache, tables, lens, new_key[keep], new_value[keep],
                       new_seq[keep], new_pos[keep], torch.zeros((0, 2), dtype=torch.int64),
                       float(D) ** -0.5)
    return inp.to(device)


@dataclass
class PrefillInputs:
    """One prompt step (K/V of the history and the prompt already in the pools)."""

    workload: Workload
    q: torch.Tensor               # [T][Hq][D] query rows of all prompts
    k_cache: torch.Tensor         # [NB][Hkv][B][D]
    v_cache: torch.Tensor
    block_tables: torch.Tensor    # int32 [S][max_blocks]
    context_lens: torch.Tensor    # int32 [S], prompts included
    q_start: torch.Tensor         # int32 [S + 1]: rows of sequence s are q_start[s] .. q_start[s+1]-1
    max_q_len: int
    scale: float

    def to(self, device) -> "PrefillInputs":
        mv = lambda t: t.to(device)  # noqa: E731
        return PrefillInputs(self.workload, mv(self.q), mv(self.k_cache), mv(self.v_cache), mv(self.block_tables),
                             mv(self.context_lens), mv(self.q_start), self.max_q_len, self.scale)


def make_prefill_inputs(w: Workload, seed: int = 0, device="cpu") -> PrefillInputs:
    """Inputs of a prompt step: context lengths as drawn, prompt lengths drawn in
    [prompt_min, prompt_max] (at most the context), random placement."""
    gen = cpu_generator(seed)
    lens = draw_lengths(w, gen)
    tables = draw_full_tables(w, gen)
    n = torch.randint(w.prompt_min, w.prompt_max + 1, (w.num_seqs,), generator=gen, dtype=torch.int64)
    n = torch.minimum(n, lens.to(torch.int64))
    q_start = torch.zeros(w.num_seqs + 1, dtype=torch.int64)
    q_start[1:] = torch.cumsum(n, 0)
    T = int(q_start[-1])
    q = randn((T, w.num_heads, w.head_dim), w.dtype, gen)
    k_cache, v_cache = draw_pools(w, gen, device, seed)
    inp = PrefillInputs(w, q, k_cache, v_cache, tables, lens, q_start.to(torch.int32), int(n.max()) if len(n) else 0,
                        float(w.head_dim) ** -0.5)
    return inp.to(device)
