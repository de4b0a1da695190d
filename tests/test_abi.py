"""The C-ABI library builds for sm_103a, loads, and exports every function the
header declares.  No compute call: this runs without a GPU."""
import ctypes

from paged_kv_cache_170_gb300 import build


def test_library_builds_loads_and_exports_header_symbols():
    path = build.build()
    lib = ctypes.CDLL(path)
    from paged_kv_cache_170_gb300 import ops  # loads the same library through the binding

    names = ops.header_functions()
    expected = {"pa_status_string", "pa_slot_mapping", "pa_write_kv", "pa_copy_blocks", "pa_decode_workspace_size",
                "pa_decode", "pa_decode_grid_size", "pa_decode_noalloc", "pa_share_plan",
                "pa_decode_shared_workspace_size", "pa_decode_shared", "pa_prefill"}
    assert expected <= set(names), sorted(expected - set(names))
    for name in names:
        assert hasattr(lib, name), f"{name} declared in include/pagedkv.h but not exported"


def test_status_strings_and_host_validation_without_gpu():
    from paged_kv_cache_170_gb300 import ops

    assert ops.lib.pa_status_string(0) == b"PA_OK"
    assert ops.lib.pa_status_string(4) == b"PA_ERR_WORKSPACE"
    # invalid host arguments are rejected before any CUDA call
    assert ops.lib.pa_write_kv(None, None, None, None, None, 1, 0, 128, 16, 10, 2, None, None) == 1
    assert ops.lib.pa_write_kv(None, None, None, None, None, 1, 8, 96, 16, 10, 2, None, None) == 1
    assert ops.lib.pa_copy_blocks(None, None, None, 1, 8, 128, 65, 10, 2, None, None) == 1
    assert ops.lib.pa_slot_mapping(None, None, 1, 1, None, None, 1, 0, 10, None, None) == 1
    assert ops.lib.pa_write_kv(None, None, None, None, None, 0, 8, 128, 16, 10, 2, None, None) == 0  # no-op


def test_product_path_does_not_import_the_oracle():
    import ast
    import os

    pkg = os.path.dirname(build.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith(".py"):
                tree = ast.parse(open(os.path.join(root, f), encoding="utf-8").read())
                for node in ast.walk(tree):
                    if isinstance(node, ast.Import):
                        assert not any(a.name.split(".")[0] == "oracle" for a in node.names), f
                    if isinstance(node, ast.ImportFrom) and node.module:
                        assert node.module.split(".")[0] != "oracle", f


def _header_signatures():
    """{name: [parameter declarations]} of every function include/pagedkv.h declares."""
    import re

    from paged_kv_cache_170_gb300 import ops

    text = open(ops.HEADER_PATH, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    sigs = {}
    for m in re.finditer(r"PA_API\s+[\w\s\*]*?\b(pa_\w+)\s*\(([^)]*)\)\s*;", text):
        params = [p.strip() for p in m.group(2).split(",") if p.strip() and p.strip() != "void"]
        sigs[m.group(1)] = params
    return sigs


def test_header_signatures_match_the_binding_and_the_recorded_boundary():
    """Every declared function has the arity the ctypes binding passes, and the
    calls of the decode step keep the parameter lists the design records
    (pa_decode without a max_context_len, its workspace sized by the head
    counts and head_dim, debug_err on the write and copy calls)."""
    from paged_kv_cache_170_gb300 import ops

    sigs = _header_signatures()
    assert set(sigs) == set(ops.header_functions())
    for name, params in sigs.items():
        fn = getattr(ops.lib, name)
        assert fn.argtypes is not None, f"{name}: the binding declares no argtypes"
        assert len(fn.argtypes) == len(params), (name, len(fn.argtypes), params)
    names = {n: [p.split()[-1].lstrip("*") for p in ps] for n, ps in sigs.items()}
    assert names["pa_decode_workspace_size"] == ["num_seqs", "num_heads", "num_kv_heads", "head_dim"]
    assert "max_context_len" not in names["pa_decode"]
    assert names["pa_decode"][:3] == ["out", "q", "k_cache"]
    assert names["pa_decode"][-3:] == ["workspace_bytes", "debug_err", "stream"]
    assert names["pa_write_kv"][-2:] == ["debug_err", "stream"]
    assert names["pa_copy_blocks"][-2:] == ["debug_err", "stream"]
    assert len(sigs["pa_decode"]) == 19 and len(sigs["pa_write_kv"]) == 13 and len(sigs["pa_copy_blocks"]) == 11
