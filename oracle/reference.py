"""Plain fp64 reference (oracle) for paged KV-cache decode attention.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this module; the product
path never does.  It shares no code with the CUDA library and imports nothing
from the product package.

Sources (pages, by title and section):
  * lihaoran.work "auto-20261007-1900", section "末块会浪费多少空间？":
    a sequence of T cached tokens with block size b needs ceil(T/b) blocks and
    leaves ceil(T/b)*b - T empty slots; T = 0 takes no block; negative sizes
    are invalid.                                            -> block_layout
  * aiqz.cc "paged-attention-mechanism", section "块表映射机制":
    pid = block_table[i], off = j mod B; lihaoran.work, section
    "块表把逻辑顺序映射到物理位置": logical block t // b, offset t % b.
                                                           -> locate, slot_of
  * aiqz.cc, section "前缀共享机制": a write into a shared block first
    allocates a new block, copies the old contents, then writes the token.
                                                    -> write_kv, copy_blocks
  * Decode: the new token attends to the whole cached history (aiqz.cc,
    section "显存痛点"); the kernel looks up the block table before reading
    the block (cf-1.com news/5879632, section 5.1).  The attention formula
    softmax(scale * q K^T) V and the grouped-query mapping
    kv_head = h // (Hq // Hkv) are not printed on the pages: they are the
    textbook definition, evaluated in float64 on the stored input values in
    logical token order.                                     -> decode
  * Prefill: the prompt's tokens enter blocks as the request arrives
    (cf-1.com news/5879632, section 3.2) and each attends to all history
    before it (aiqz.cc, section "显存痛点"); causally, prompt token i sees
    the history and prompt tokens 0 .. i.               -> prefill

Layouts: q/out [S][Hq][D]; K/V pools [NB][Hkv][B][D]; block_tables int32
[S][max_blocks]; context_lens int32 [S]; slot_mapping int64 [T]; copy pairs
int64 [P][2] (src, dst).
"""
from __future__ import annotations

import math

import numpy as np
import torch


def block_layout(tokens: int, block_size: int) -> tuple[int, int]:
    """(blocks, unused slots) for ``tokens`` cached tokens in blocks of ``block_size``."""
    if tokens < 0 or block_size <= 0:
        raise ValueError("invalid size")
    blocks = -(-tokens // block_size)
    return blocks, blocks * block_size - tokens


def locate(table_row, t: int, block_size: int) -> tuple[int, int]:
    """Token position ``t`` -> (physical block id, offset inside the block)."""
    if t < 0 or block_size <= 0:
        raise ValueError("invalid position")
    logical = t // block_size
    if logical >= len(table_row):
        raise IndexError("position beyond the block table")
    return int(table_row[logical]), t % block_size


def slot_of(table_row, t: int, block_size: int) -> int:
    """Flat slot index pid * B + off of token position ``t``."""
    pid, off = locate(table_row, t, block_size)
    return pid * block_size + off


def kv_head(h: int, num_heads: int, num_kv_heads: int) -> int:
    """KV head read by query head ``h``: contiguous groups of Hq/Hkv heads."""
    return h // (num_heads // num_kv_heads)


def _f64(x: torch.Tensor) -> np.ndarray:
    return x.detach().to("cpu").to(torch.float64).numpy()


def slot_mapping(block_tables, token_seq, token_pos, block_size: int) -> np.ndarray:
    """Slots of new tokens: token i belongs to sequence token_seq[i] at position token_pos[i]."""
    tables = np.asarray(block_tables)
    out = np.empty(len(token_seq), dtype=np.int64)
    for i, (s, t) in enumerate(zip(np.asarray(token_seq).tolist(), np.asarray(token_pos).tolist())):
        out[i] = slot_of(tables[s], t, block_size)
    return out


def write_kv(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor,
             v_cache: torch.Tensor, slots) -> None:
    """In place: row [i][h] of key/value goes to pool[slot // B][h][slot % B]; slot < 0 skips."""
    B = k_cache.shape[2]
    NB = k_cache.shape[0]
    for i, slot in enumerate(np.asarray(slots).tolist()):
        if slot < 0:
            continue
        if slot >= NB * B:
            raise IndexError("slot outside the pool")
        pid, off = divmod(slot, B)
        k_cache[pid, :, off, :] = key[i]
        v_cache[pid, :, off, :] = value[i]


def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, pairs) -> None:
    """In place, in order: whole block dst <- block src, for K and V."""
    NB = k_cache.shape[0]
    for src, dst in np.asarray(pairs, dtype=np.int64).reshape(-1, 2).tolist():
        if not (0 <= src < NB and 0 <= dst < NB):
            raise IndexError("block id outside the pool")
        k_cache[dst] = k_cache[src].clone()
        v_cache[dst] = v_cache[src].clone()


def decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
           block_tables, context_lens, scale: float) -> np.ndarray:
    """float64 [S][Hq][D]: softmax(scale * q K^T) V through the block table.

    Sequences with no cached token give a zero row.
    """
    S, Hq, D = q.shape
    Hkv, B = k_cache.shape[1], k_cache.shape[2]
    qd, kd, vd = _f64(q), _f64(k_cache), _f64(v_cache)
    tables = np.asarray(block_tables)
    lens = np.asarray(context_lens).tolist()
    out = np.zeros((S, Hq, D), dtype=np.float64)
    for s in range(S):
        L = int(lens[s])
        if L == 0:
            continue
        where = [locate(tables[s], t, B) for t in range(L)]
        pids = np.array([w[0] for w in where], dtype=np.int64)
        offs = np.array([w[1] for w in where], dtype=np.int64)
        for h in range(Hq):
            g = kv_head(h, Hq, Hkv)
            K = kd[pids, g, offs, :]          # [L][D], logical order
            V = vd[pids, g, offs, :]
            x = scale * (K @ qd[s, h])        # [L]
            w = np.exp(x - x.max())
            out[s, h] = (w @ V) / w.sum()
    return out


def prefill(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
            block_tables, context_lens, q_start, scale: float) -> np.ndarray:
    """float64 [T][Hq][D] prompt attention through the block table.

    Sequence s owns query rows q_start[s] .. q_start[s+1]-1: the last n of its
    context_lens[s] positions.  Row i, at position p = L - n + i, attends to
    tokens 0 .. p (the history, then the prompt up to itself).
    """
    T, Hq, D = q.shape
    Hkv, B = k_cache.shape[1], k_cache.shape[2]
    qd, kd, vd = _f64(q), _f64(k_cache), _f64(v_cache)
    tables = np.asarray(block_tables)
    lens = np.asarray(context_lens).tolist()
    qs = np.asarray(q_start).tolist()
    out = np.zeros((T, Hq, D), dtype=np.float64)
    for s in range(len(lens)):
        L, n = int(lens[s]), int(qs[s + 1] - qs[s])
        if n == 0:
            continue
        addr = [locate(tables[s], tok, B) for tok in range(L)]
        pid = np.array([a[0] for a in addr], dtype=np.int64)
        off = np.array([a[1] for a in addr], dtype=np.int64)
        for i in range(n):
            p = L - n + i      # this query row's position in the sequence
            end = p + 1        # it sees tokens 0 .. p
            for h in range(Hq):
                g = kv_head(h, Hq, Hkv)
                Kc = kd[pid[:end], g, off[:end], :]
                Vc = vd[pid[:end], g, off[:end], :]
                z = scale * (Kc @ qd[qs[s] + i, h])
                e = np.exp(z - np.max(z))
                out[qs[s] + i, h] = (e @ Vc) / np.sum(e)
    return out


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)
