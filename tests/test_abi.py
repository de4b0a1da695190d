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
