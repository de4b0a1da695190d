"""Thin Python binding of libpagedkv.so (the C ABI in include/pagedkv.h).

Argument marshalling only: every function checks devices/dtypes/shapes of the
torch tensors, passes raw device pointers and the current CUDA stream to the
C entry point of the same name, and raises ``PagedKVError`` on a non-OK
status.  All arithmetic runs in the library's CUDA kernels; there is no other
code path.  Importing this module loads the library and raises if it has not
been built (``python -m paged_kv_cache_170_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libpagedkv.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "pagedkv.h")

PA_OK = 0
_DTYPES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
DEVERR_BITS = {1: "BLOCK_ID", 2: "SLOT", 4: "CONTEXT", 8: "TIMEOUT", 16: "POSITION", 32: "LAYOUT",
               256: "DEBUG_SMEM_RANGE", 512: "DEBUG_TMA_BOX", 1024: "DEBUG_GLOBAL_RANGE", 2048: "DEBUG_BARRIER_PHASE"}


class PagedKVError(RuntimeError):
    pass


def _load(path: str = LIB_PATH) -> ctypes.CDLL:
    """The library at ``path`` with every entry point's argument types set."""
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python -m paged_kv_cache_170_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    sig = {
        "pa_slot_mapping": [vp, vp, i32, i32, vp, vp, i64, i32, i64, vp, vp],
        "pa_write_kv": [vp, vp, vp, vp, vp, i64, i32, i32, i32, i64, i32, vp, vp],
        "pa_copy_blocks": [vp, vp, vp, i64, i32, i32, i32, i64, i32, vp, vp],
        "pa_decode": [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i64, f32, i32, vp, sz, vp, vp],
        "pa_decode_noalloc": [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i64, f32, i32, vp, vp],
        "pa_write_decode": [vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i64, f32, i32, vp, sz,
                            vp, vp],
        "pa_share_plan": [vp, i32, vp, i32, i32, i32, i32, i32, vp, sz, ctypes.POINTER(sz)],
        "pa_decode_shared": [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i64, f32, i32, vp, vp, vp, sz,
                             vp, vp],
        "pa_prefill": [vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32, i64, f32, i32, vp, vp],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = i32
    lib.pa_decode_workspace_size.argtypes = [i32, i32, i32, i32]
    lib.pa_decode_workspace_size.restype = sz
    lib.pa_decode_shared_workspace_size.argtypes = [vp, i32, i32, i32, i32]
    lib.pa_decode_shared_workspace_size.restype = sz
    lib.pa_decode_grid_size.argtypes = []
    lib.pa_decode_grid_size.restype = i32
    lib.pa_status_string.argtypes = [i32]
    lib.pa_status_string.restype = ctypes.c_char_p
    return lib


lib = _load()


def header_functions() -> list[str]:
    """Names of the functions include/pagedkv.h declares."""
    with open(HEADER_PATH, encoding="utf-8") as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:PA_API\s+)?(?:pa_status|size_t|int|const char \*)\s*\*?\s*(pa_\w+)\s*\(", text, re.M)))


def _check(status: int, what: str) -> None:
    if status != PA_OK:
        raise PagedKVError(f"{what}: {lib.pa_status_string(status).decode()}")


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _need(t: torch.Tensor, name: str, dtype=None, ndim=None, device=None) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


def new_error_word(device) -> torch.Tensor:
    """A zeroed device int32 for the kernels' error bits (``debug_err``)."""
    return torch.zeros(1, dtype=torch.int32, device=device)


def error_names(word: int) -> list[str]:
    return [name for bit, name in DEVERR_BITS.items() if word & bit]


def pa_slot_mapping(block_tables: torch.Tensor, token_seq: torch.Tensor, token_pos: torch.Tensor,
                    block_size: int, num_blocks: int, out: Optional[torch.Tensor] = None,
                    err: Optional[torch.Tensor] = None) -> torch.Tensor:
    dev = block_tables.device
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(token_seq, "token_seq", torch.int32, 1, dev)
    _need(token_pos, "token_pos", torch.int32, 1, dev)
    n = token_seq.numel()
    if token_pos.numel() != n:
        raise ValueError("token_seq and token_pos differ in length")
    if out is None:
        out = torch.empty(n, dtype=torch.int64, device=dev)
    _need(out, "out", torch.int64, 1, dev)
    S, width = block_tables.shape
    _check(lib.pa_slot_mapping(out.data_ptr(), block_tables.data_ptr(), width, S, token_seq.data_ptr(),
                               token_pos.data_ptr(), n, block_size, num_blocks, _ptr(err), _stream(dev)),
           "pa_slot_mapping")
    return out


def _cache_shape(k_cache: torch.Tensor, v_cache: torch.Tensor):
    _need(k_cache, "k_cache", None, 4)
    _need(v_cache, "v_cache", k_cache.dtype, 4, k_cache.device)
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache differ in shape")
    if k_cache.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {k_cache.dtype}")
    return k_cache.shape  # NB, Hkv, B, D


def pa_write_kv(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                slot_mapping: torch.Tensor, err: Optional[torch.Tensor] = None) -> None:
    NB, Hkv, B, D = _cache_shape(k_cache, v_cache)
    dev = k_cache.device
    _need(key, "key", k_cache.dtype, 3, dev)
    _need(value, "value", k_cache.dtype, 3, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    T = key.shape[0]
    if key.shape != (T, Hkv, D) or value.shape != key.shape or slot_mapping.numel() != T:
        raise ValueError("key/value must be [T][Hkv][D] with one slot per token")
    _check(lib.pa_write_kv(key.data_ptr(), value.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                           slot_mapping.data_ptr(), T, Hkv, D, B, NB, _DTYPES[k_cache.dtype], _ptr(err),
                           _stream(dev)), "pa_write_kv")


def pa_copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, pairs: torch.Tensor,
                   err: Optional[torch.Tensor] = None) -> None:
    NB, Hkv, B, D = _cache_shape(k_cache, v_cache)
    dev = k_cache.device
    _need(pairs, "pairs", torch.int64, None, dev)
    if pairs.numel() % 2:
        raise ValueError("pairs must be [P][2]")
    _check(lib.pa_copy_blocks(k_cache.data_ptr(), v_cache.data_ptr(), pairs.data_ptr(), pairs.numel() // 2, Hkv,
                              D, B, NB, _DTYPES[k_cache.dtype], _ptr(err), _stream(dev)), "pa_copy_blocks")


def pa_decode_workspace_size(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int) -> int:
    n = lib.pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim)
    if n == 0:
        raise PagedKVError("pa_decode_workspace_size: invalid shape or no CUDA device")
    return int(n)


def pa_decode_grid_size() -> int:
    return int(lib.pa_decode_grid_size())


def new_workspace(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int, device) -> torch.Tensor:
    """A decode workspace, zero-filled as pa_decode requires before first use."""
    n = pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def _decode_args(q, k_cache, v_cache, block_tables, context_lens, out, workspace, with_workspace=True):
    """Checks of a decode call's tensors; ``out`` and (with_workspace) the
    workspace are allocated when not given."""
    NB, Hkv, B, D = _cache_shape(k_cache, v_cache)
    dev = k_cache.device
    _need(q, "q", k_cache.dtype, 3, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    S, Hq, Dq = q.shape
    if Dq != D or block_tables.shape[0] != S or context_lens.numel() != S:
        raise ValueError("q [S][Hq][D], block_tables [S][*], context_lens [S] disagree")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", q.dtype, 3, dev)
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if with_workspace:
        if workspace is None:
            workspace = new_workspace(S, Hq, Hkv, D, dev)
        _need(workspace, "workspace", torch.uint8, 1, dev)
    return NB, Hkv, B, D, S, Hq, out, workspace


def pa_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
              context_lens: torch.Tensor, scale: float, out: Optional[torch.Tensor] = None,
              workspace: Optional[torch.Tensor] = None, err: Optional[torch.Tensor] = None) -> torch.Tensor:
    NB, Hkv, B, D, S, Hq, out, ws = _decode_args(q, k_cache, v_cache, block_tables, context_lens, out, workspace)
    _check(lib.pa_decode(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                         block_tables.data_ptr(), block_tables.shape[1], context_lens.data_ptr(), S, Hq, Hkv, D, B,
                         NB, float(scale), _DTYPES[q.dtype], ws.data_ptr(), ws.numel(), _ptr(err),
                         _stream(q.device)), "pa_decode")
    return out


def pa_write_decode(q: torch.Tensor, new_key: torch.Tensor, new_value: torch.Tensor, k_cache: torch.Tensor,
                    v_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                    out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                    err: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Each sequence's new token (new_key / new_value [S][Hkv][D], at position
    context_lens[s] - 1) written into its slot, then decode attention: two
    launches, the decode allowed to start while the write runs."""
    NB, Hkv, B, D, S, Hq, out, ws = _decode_args(q, k_cache, v_cache, block_tables, context_lens, out, workspace)
    for name, t in (("new_key", new_key), ("new_value", new_value)):
        _need(t, name, k_cache.dtype, 3, k_cache.device)
        if tuple(t.shape) != (S, Hkv, D):
            raise ValueError(f"{name} must be [num_seqs][num_kv_heads][head_dim]")
    _check(lib.pa_write_decode(out.data_ptr(), q.data_ptr(), new_key.data_ptr(), new_value.data_ptr(),
                               k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(), block_tables.shape[1],
                               context_lens.data_ptr(), S, Hq, Hkv, D, B, NB, float(scale), _DTYPES[q.dtype],
                               ws.data_ptr(), ws.numel(), _ptr(err), _stream(q.device)), "pa_write_decode")
    return out


def pa_decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                      context_lens: torch.Tensor, scale: float, out: Optional[torch.Tensor] = None,
                      err: Optional[torch.Tensor] = None) -> torch.Tensor:
    """pa_decode without a workspace, for callers that cannot allocate device
    memory: the library keeps the scratch in a static 4 MiB device array.
    ``out`` is still the caller's (allocated here only when not given)."""
    NB, Hkv, B, D, S, Hq, out, _ = _decode_args(q, k_cache, v_cache, block_tables, context_lens, out, None,
                                                with_workspace=False)
    dev = q.device
    _check(lib.pa_decode_noalloc(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                 block_tables.data_ptr(), block_tables.shape[1], context_lens.data_ptr(), S, Hq, Hkv,
                                 D, B, NB, float(scale), _DTYPES[q.dtype], _ptr(err), _stream(dev)),
           "pa_decode_noalloc")
    return out


# Field order of the plan header (csrc/pa_share_plan.h); each array field is
# the array's offset in ints from the start of the plan.
PLAN_FIELDS = ["magic", "total_ints", "num_seqs", "num_groups", "num_units", "num_pieces", "nctas", "group_size",
               "num_kv_heads", "block_size", "max_blocks", "total_members", "total_memberships", "g_moff",
               "g_members", "g_b0", "g_b1", "g_ubase", "g_passes", "u_group", "u_kvh", "u_pass", "u_poff", "p_unit",
               "p_t0", "p_t1", "c_poff", "s_start", "s_moff", "s_mgroup", "s_midx", "own_tiles", "num_shared_groups",
               "g_prows", "c_opoff", "p_desc", "num_tc_items", "t_items", "r_off", "r_rec", "tc_chunk_steps",
               "t_qrow", "t_blk", "t_blk_stride"]


def share_plan(block_tables: torch.Tensor, context_lens: torch.Tensor, block_size: int, num_heads: int,
               num_kv_heads: int, nctas: Optional[int] = None) -> torch.Tensor:
    """pa_share_plan on host copies of the tables: the plan as a CPU int32
    tensor (copy it to the device for pa_decode_shared)."""
    tables = block_tables.detach().to("cpu", torch.int32).contiguous()
    lens = context_lens.detach().to("cpu", torch.int32).contiguous()
    S, width = tables.shape
    if lens.numel() != S:
        raise ValueError("context_lens and block_tables differ in rows")
    n = lib.pa_decode_grid_size() if nctas is None else int(nctas)
    need = ctypes.c_size_t(0)
    _check(lib.pa_share_plan(tables.data_ptr(), width, lens.data_ptr(), S, block_size, num_heads, num_kv_heads, n,
                             None, 0, ctypes.byref(need)), "pa_share_plan")
    plan = torch.zeros(int(need.value), dtype=torch.int32)
    _check(lib.pa_share_plan(tables.data_ptr(), width, lens.data_ptr(), S, block_size, num_heads, num_kv_heads, n,
                             plan.data_ptr(), plan.numel(), ctypes.byref(need)), "pa_share_plan")
    return plan


def plan_fields(plan: torch.Tensor) -> dict:
    """The plan's header as a dict, and its arrays (numpy) under their names."""
    p = plan.numpy()
    hdr = {k: int(p[i]) for i, k in enumerate(PLAN_FIELDS)}
    n = {"g_moff": hdr["num_groups"] + 1, "g_members": hdr["total_members"], "g_b0": hdr["num_groups"],
         "g_b1": hdr["num_groups"], "g_ubase": hdr["num_groups"], "g_passes": hdr["num_groups"],
         "u_group": hdr["num_units"], "u_kvh": hdr["num_units"], "u_pass": hdr["num_units"],
         "u_poff": hdr["num_units"] + 1, "p_unit": hdr["num_pieces"], "p_t0": hdr["num_pieces"],
         "p_t1": hdr["num_pieces"], "c_poff": hdr["nctas"] + 1, "s_start": hdr["num_seqs"],
         "s_moff": hdr["num_seqs"] + 1, "s_mgroup": hdr["total_memberships"], "s_midx": hdr["total_memberships"],
         "g_prows": hdr["num_groups"], "c_opoff": hdr["nctas"] + 1, "p_desc": hdr["num_pieces"] * 12,
         "t_items": hdr["num_tc_items"] * 12, "t_qrow": hdr["num_tc_items"] * 128,
         "t_blk": hdr["num_tc_items"] * hdr["t_blk_stride"]}
    out = dict(hdr)
    for k, cnt in n.items():
        out[k + "_arr"] = p[hdr[k]:hdr[k] + cnt]
    # each output row's record list: r_off[S * Hq + 1] ends where r_rec starts
    out["r_off_arr"] = p[hdr["r_off"]:hdr["r_rec"]]
    out["r_rec_arr"] = p[hdr["r_rec"]:hdr["r_rec"] + int(out["r_off_arr"][-1])] if len(out["r_off_arr"]) else p[:0]
    return out


def new_shared_workspace(plan_host: torch.Tensor, num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int,
                         device) -> torch.Tensor:
    nbytes = lib.pa_decode_shared_workspace_size(plan_host.data_ptr(), num_seqs, num_heads, num_kv_heads, head_dim)
    if nbytes == 0:
        raise PagedKVError("pa_decode_shared_workspace_size: invalid arguments")
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


def pa_decode_shared(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                     context_lens: torch.Tensor, scale: float, plan_host: torch.Tensor, plan_dev: torch.Tensor,
                     out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                     err: Optional[torch.Tensor] = None) -> torch.Tensor:
    """pa_decode reading each shared block once per group of sharers, with a
    plan from ``share_plan`` (host copy and a device copy of it)."""
    if plan_host.device.type != "cpu" or plan_host.dtype != torch.int32 or not plan_host.is_contiguous():
        raise ValueError("plan_host must be a contiguous CPU int32 tensor")
    if workspace is None:
        S, Hq, D = q.shape
        workspace = new_shared_workspace(plan_host, S, Hq, k_cache.shape[1], D, q.device)
    NB, Hkv, B, D, S, Hq, out, workspace = _decode_args(q, k_cache, v_cache, block_tables, context_lens, out,
                                                        workspace)
    _need(plan_dev, "plan_dev", torch.int32, 1, q.device)
    if plan_dev.numel() != plan_host.numel():
        raise ValueError("plan_dev and plan_host differ in size")
    _check(lib.pa_decode_shared(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                block_tables.data_ptr(), block_tables.shape[1], context_lens.data_ptr(), S, Hq, Hkv,
                                D, B, NB, float(scale), _DTYPES[q.dtype], plan_host.data_ptr(), plan_dev.data_ptr(),
                                workspace.data_ptr(), workspace.numel(), _ptr(err), _stream(q.device)),
           "pa_decode_shared")
    return out


def pa_prefill(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
               context_lens: torch.Tensor, q_start: torch.Tensor, max_q_len: int, scale: float,
               out: Optional[torch.Tensor] = None, err: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Prompt attention: q [T][Hq][D], the query rows of sequence s being
    q[q_start[s]:q_start[s+1]] (the last positions of its context)."""
    NB, Hkv, B, D = _cache_shape(k_cache, v_cache)
    dev = k_cache.device
    _need(q, "q", k_cache.dtype, 3, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    _need(q_start, "q_start", torch.int32, 1, dev)
    S = context_lens.numel()
    if block_tables.shape[0] != S or q_start.numel() != S + 1 or q.shape[2] != D:
        raise ValueError("q [T][Hq][D], block_tables [S][*], context_lens [S], q_start [S+1] disagree")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", q.dtype, 3, dev)
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    _check(lib.pa_prefill(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                          block_tables.data_ptr(), block_tables.shape[1], context_lens.data_ptr(), q_start.data_ptr(),
                          S, int(max_q_len), q.shape[1], Hkv, D, B, NB, float(scale), _DTYPES[q.dtype], _ptr(err),
                          _stream(dev)), "pa_prefill")
    return out


def decode_step(inp, out=None, workspace=None, slots=None, err=None) -> torch.Tensor:
    """One whole decode step on resident inputs: copy-on-write block copies,
    slot lookup of the new tokens, their K/V write, then decode attention."""
    if inp.copy_pairs.numel():
        pa_copy_blocks(inp.k_cache, inp.v_cache, inp.copy_pairs, err)
    if inp.new_seq.numel():
        B = inp.k_cache.shape[2]
        slots = pa_slot_mapping(inp.block_tables, inp.new_seq, inp.new_pos, B, inp.k_cache.shape[0], slots, err)
        pa_write_kv(inp.new_key, inp.new_value, inp.k_cache, inp.v_cache, slots, err)
    return pa_decode(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale, out,
                     workspace, err)
