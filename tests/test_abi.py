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

    for code in range(0, 12):
        assert pa._lib.pa_status_str(code)


def test_prefill_host_checks_run_before_any_launch():
    """Argument errors of pa_prefill_attention come back from the host checks (no GPU needed)."""
    import paged_kv_cache_280_gb300 as pa

    fake = ctypes.c_void_p(1 << 20)  # 16-byte aligned, never dereferenced
    args = lambda dt, hd, bs: (fake, fake, fake, fake, fake, 4, fake, fake, 2, 10, 8, 8, 2, hd, bs, 100, 0.1, dt,  # noqa: E731
                               None, None)
    assert pa._lib.pa_prefill_attention(*args(pa.PA_F32, 128, 16)) == 2  # PA_ERR_UNSUPPORTED: fp32
    assert pa._lib.pa_prefill_attention(*args(pa.PA_BF16, 96, 16)) == 2  # head_dim 96
    assert pa._lib.pa_prefill_attention(*args(pa.PA_BF16, 128, 8)) == 2  # block_size 8
    bad = list(args(pa.PA_BF16, 128, 16))
    bad[1] = ctypes.c_void_p((1 << 20) + 2)  # misaligned q
    assert pa._lib.pa_prefill_attention(*bad) == 1  # PA_ERR_INVALID_ARG
    for scale in (0.0, -0.1):  # the tensor-core prefill needs a positive scale
        bad = list(args(pa.PA_BF16, 128, 16))
        bad[16] = scale
        assert pa._lib.pa_prefill_attention(*bad) == 1


def test_swap_host_checks_run_before_any_launch():
    import paged_kv_cache_280_gb300 as pa

    fake = ctypes.c_void_p(1 << 20)
    ok_args = [fake, fake, fake, 4, fake, fake, 8, 128, 16, 100, pa.PA_BF16, None, None]
    assert pa._lib.pa_swap_out(*ok_args[:8], 12, *ok_args[9:]) == 2  # block_size 12: unsupported
    bad = list(ok_args)
    bad[4] = ctypes.c_void_p((1 << 20) + 8)  # misaligned store
    assert pa._lib.pa_swap_out(*bad) == 1
    assert pa._lib.pa_swap_in(*ok_args[:3], 0, *ok_args[4:]) == 0  # nothing to copy


def test_wait_limit_knob_checks_its_argument():
    """The failure-detection testing aid runs on the host: above the 2 s default is refused, 0 restores it."""
    import pytest
    import paged_kv_cache_280_gb300 as pa

    with pytest.raises(pa.PAError):
        pa.pa_debug_set_wait_limit_ns(3_000_000_000)
    pa.pa_debug_set_wait_limit_ns(0)


def test_merge_mode_knob_checks_its_argument():
    import pytest
    import paged_kv_cache_280_gb300 as pa

    for bad in (-1, 3):
        with pytest.raises(pa.PAError):
            pa.pa_debug_set_merge_mode(bad)
    pa.pa_debug_set_merge_mode(pa.MERGE_AUTO)


def test_seg_units_knob_checks_its_argument():
    import pytest
    import paged_kv_cache_280_gb300 as pa

    for bad in (-1, 4097):
        with pytest.raises(pa.PAError):
            pa.pa_debug_set_seg_units(bad)
    pa.pa_debug_set_seg_units(0)


def test_wave_skew_knob_checks_its_argument():
    import pytest
    import paged_kv_cache_280_gb300 as pa

    for bad in (-2, 9):
        with pytest.raises(pa.PAError):
            pa.pa_debug_set_wave_skew(bad)
    pa.pa_debug_set_wave_skew(-1)
