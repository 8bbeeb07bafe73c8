"""The C-ABI library loads on a host without a GPU and exports every symbol
include/pa.h declares; host-only calls behave as documented."""
import ctypes as C
import os
import re

import pytest

from conftest import ROOT


def declared_functions():
    src = open(os.path.join(ROOT, "include", "pa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_the_hot_path_calls():
    names = declared_functions()
    for n in ("pa_reshape_and_cache", "pa_decode", "pa_copy_blocks", "pa_decode_workspace_size",
              "pa_alloc_create", "pa_alloc_append_slot", "pa_alloc_fork"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from paged_kv_cache_142_gb300 import _lib
    names = declared_functions()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert sorted(_lib.SIGNATURES) == names  # the binding declares exactly the header's calls


def test_status_strings_and_version(lib):
    assert lib.pa_status_string(0) == b"PA_OK"
    assert lib.pa_status_string(4) == b"PA_ERR_OOM"
    assert b"sm_103a" in lib.pa_version()


def test_workspace_size_plan_is_host_only(lib):
    # split-K workspace for a long context is larger than for a short one
    small = lib.pa_decode_workspace_size(8, 64, 8, 128, 16, 1, 256, 0)
    big = lib.pa_decode_workspace_size(8, 64, 8, 128, 16, 1, 32768, 0)
    assert 0 < small < big
    # 8 seqs * 8 kv heads * 8 partitions of 4096 tokens * 8 heads * (128 + 2)
    # floats, plus header and counters
    assert big >= 8 * 8 * 8 * 8 * 130 * 4
    # unsupported group size -> 0
    assert lib.pa_decode_workspace_size(1, 48, 2, 128, 16, 1, 100, 0) == 0
    pt = C.c_int32(0)
    # bf16, head_dim 128: tensor-core kernel, 4096-token partitions past 4096
    # tokens of context and 2048 up to it, when the (sequence, kv head,
    # partition) items cover every SM twice ...
    st = lib.pa_decode_plan(8, 64, 8, 128, 16, 1, 32768, 0, C.byref(pt), None)
    assert st == 0 and pt.value == 4096
    st = lib.pa_decode_plan(256, 64, 8, 128, 16, 1, 4096, 0, C.byref(pt), None)
    assert st == 0 and pt.value == 2048
    # ... halved down to 256 tokens while they do not
    st = lib.pa_decode_plan(2, 64, 8, 128, 16, 1, 32768, 0, C.byref(pt), None)
    assert st == 0 and pt.value == 1024
    st = lib.pa_decode_plan(8, 64, 8, 128, 16, 1, 4096, 0, C.byref(pt), None)
    assert st == 0 and pt.value == 512
    st = lib.pa_decode_plan(1, 64, 8, 128, 16, 1, 4096, 0, C.byref(pt), None)
    assert st == 0 and pt.value == 256
    # fp32: CUDA-core kernel, 256-token partitions
    st = lib.pa_decode_plan(8, 64, 8, 128, 16, 0, 32768, 0, C.byref(pt), None)
    assert st == 0 and pt.value == 256
    # an explicit partition is rounded up to the 128-token tile
    st = lib.pa_decode_plan(8, 64, 8, 128, 16, 1, 32768, 200, C.byref(pt), None)
    assert st == 0 and pt.value == 256


def test_argument_errors_return_before_any_launch(lib):
    from paged_kv_cache_142_gb300 import _lib as L
    # bad block size / head_dim / dtype are rejected on the host
    assert lib.pa_reshape_and_cache(None, None, 1, None, None, None, 8, 12, 2, 128, 1, None) == L.PA_ERR_UNSUPPORTED
    assert lib.pa_copy_blocks(None, None, 8, 16, 2, 128, 7, None, 1, None) == L.PA_ERR_INVALID_ARG
    assert lib.pa_reshape_and_cache(None, None, 0, None, None, None, 8, 16, 2, 128, 1, None) == L.PA_OK
    # missing pointers with work to do
    assert lib.pa_reshape_and_cache(None, None, 3, None, None, None, 8, 16, 2, 128, 1, None) == L.PA_ERR_INVALID_ARG
    # num_q_heads not a multiple of num_kv_heads
    rc = lib.pa_decode(None, 0, None, 2, 6, None, None, 8, 16, 4, 128, 1, None, 4, None, 64,
                       1.0, 0, None, 0, None)
    assert rc == L.PA_ERR_INVALID_ARG
    # table too short for max_context_len
    rc = lib.pa_decode(None, 0, None, 2, 8, None, None, 8, 16, 4, 128, 1, None, 2, None, 64,
                       1.0, 0, None, 0, None)
    assert rc == L.PA_ERR_INVALID_ARG


def test_plain_c_program_uses_the_host_calls(lib, tmp_path):
    """include/pa.h is usable from C11 alone: a C program drives the block
    allocator and SHA-256 through the library, with no Python in between."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    from paged_kv_cache_142_gb300 import _lib as L
    libdir = os.path.dirname(L.LIB_PATH)
    exe = tmp_path / "c_abi_host"
    here = os.path.dirname(os.path.abspath(__file__))
    build = subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(here, "..", "include"),
                            os.path.join(here, "c_abi_host.c"), "-o", str(exe), "-L", libdir, "-lpa_gb300",
                            f"-Wl,-rpath,{libdir}"], capture_output=True, text=True)
    assert build.returncode == 0, build.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0 and run.stdout.strip() == "ok", (run.returncode, run.stderr)


def test_checked_calls_need_a_status_word(lib):
    from paged_kv_cache_142_gb300 import _lib as L
    # the checked append and copy require their status word (before any launch)
    assert lib.pa_reshape_and_cache_checked(None, None, 3, None, None, None, 8, 16, 2, 128, 1, None,
                                            None) == L.PA_ERR_INVALID_ARG
    assert lib.pa_copy_blocks_checked(None, None, 8, 16, 2, 128, 1, None, 2, None, None) == L.PA_ERR_INVALID_ARG
    # the no-alloc status read needs somewhere to put it
    assert lib.pa_decode_no_alloc_error(None, None) == L.PA_ERR_INVALID_ARG


def test_kv_per_item_setting_shapes_the_plan(lib):
    """The work-item setting is validated, and it changes the workspace the
    plan needs (one merge counter per item row) where two kv heads can pair."""
    from paged_kv_cache_142_gb300 import _lib as L
    assert lib.pa_set_decode_kv_per_item(3) == L.PA_ERR_INVALID_ARG
    assert lib.pa_set_decode_kv_per_item(-1) == L.PA_ERR_INVALID_ARG
    try:
        sizes = {}
        for kh in (1, 2):
            assert lib.pa_set_decode_kv_per_item(kh) == L.PA_OK
            sizes[kh] = lib.pa_decode_workspace_size(256, 32, 8, 128, 16, 1, 4096, 0)
        assert sizes[1] > sizes[2] > 0  # 2048 rows of counters against 1024
        # a shape that cannot pair (odd kv heads) plans the same either way
        odd = []
        for kh in (1, 2):
            lib.pa_set_decode_kv_per_item(kh)
            odd.append(lib.pa_decode_workspace_size(256, 24, 3, 128, 16, 1, 4096, 0))
        assert odd[0] == odd[1]
    finally:
        lib.pa_set_decode_kv_per_item(0)
