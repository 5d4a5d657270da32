"""The C-ABI library loads on a machine without a GPU and exports every symbol include/pa.h declares."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    with open(os.path.join(ROOT, "include", "pa.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\**\s*(pa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_hot_path():
    names = declared_functions()
    for required in ("pa_reshape_and_cache", "pa_copy_blocks", "pa_decode_attention", "pa_decode_workspace_bytes",
                     "pa_alloc_create", "pa_seq_append", "pa_append_batch", "pa_seq_fork", "pa_seq_free"):
        assert required in names


def test_library_exports_every_declared_symbol():
    import paged_kv_cache_280_gb300 as pa

    lib = ctypes.CDLL(pa.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert pa.abi_version() == 1


def test_status_strings():
    import paged_kv_cache_280_gb300 as pa

    for code in range(0, 11):
        assert pa._lib.pa_status_str(code)
