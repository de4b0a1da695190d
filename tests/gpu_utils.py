"""Helpers shared by the GPU parity tests: the oracle's view of a decode step
and the tolerance checks (fp16/bf16: max abs 2e-3 and max rel 1e-2; fp32:
abs 1e-5 + rel 1e-4)."""
from __future__ import annotations

import numpy as np
import torch

from oracle import native, reference


def to_cpu(inp):
    return inp.to("cpu")


def oracle_step(inp_cpu, seqs=None):
    """Copy-on-write copies, slot lookup, K/V write, then decode, all on the
    CPU oracle.  Returns (slots, k_cache, v_cache, out[float64]); ``seqs``
    limits the decode to a subset of sequences (rows of ``out`` follow it)."""
    kc, vc = inp_cpu.k_cache.clone(), inp_cpu.v_cache.clone()
    if inp_cpu.copy_pairs.numel():
        native.copy_blocks(kc, vc, inp_cpu.copy_pairs.numpy())
    B = kc.shape[2]
    tables = inp_cpu.block_tables.numpy()
    slots = native.slot_mapping(tables, inp_cpu.new_seq.numpy(), inp_cpu.new_pos.numpy(), B)
    if len(slots):
        native.write_kv(inp_cpu.new_key, inp_cpu.new_value, kc, vc, slots)
    lens = inp_cpu.context_lens.numpy()
    q = inp_cpu.q
    if seqs is not None:
        sel = np.asarray(seqs)
        q, tables, lens = q[torch.as_tensor(sel)], tables[sel], lens[sel]
    out = native.decode(q, kc, vc, tables, lens, inp_cpu.scale)
    return slots, kc, vc, out


def attention_errors(got: torch.Tensor, ref: np.ndarray):
    g = got.detach().float().cpu().double().numpy()
    err = np.abs(g - ref)
    big = np.abs(ref) >= 1e-2
    max_abs = float(err.max()) if err.size else 0.0
    max_rel = float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0
    return err, max_abs, max_rel


def assert_attention_close(got: torch.Tensor, ref: np.ndarray, strict: bool = True) -> dict:
    """strict: the workload bar (max abs <= 2e-3 and max rel <= 1e-2 over
    |ref| >= 1e-2).  Otherwise each element needs abs <= 2e-3 or rel <= 1e-2
    (a bf16 rounding of a value above 1 alone exceeds 2e-3)."""
    assert not torch.isnan(got).any(), "NaN in output"
    err, max_abs, max_rel = attention_errors(got, ref)
    if got.dtype == torch.float32:
        bad = err > 1e-5 + 1e-4 * np.abs(ref)
        assert not bad.any(), f"fp32: {bad.sum()} elements off, max abs {max_abs:.3g}"
    elif strict:
        assert max_abs <= 2e-3 and max_rel <= 1e-2, f"max abs {max_abs:.3g}, max rel {max_rel:.3g}"
    else:
        bad = (err > 2e-3) & (err > 1e-2 * np.abs(ref))
        assert not bad.any(), f"{bad.sum()} elements off; max abs {max_abs:.3g}, max rel {max_rel:.3g}"
    return {"max_abs": max_abs, "max_rel": max_rel}


def valid_blocks(lens, B):
    return [reference.block_layout(int(L), B)[0] for L in lens]

