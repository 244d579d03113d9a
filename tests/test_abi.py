"""The C-ABI library loads, exports every symbol the header declares, and
rejects bad arguments on the host (no GPU needed: nothing here launches)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "zr.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(zr_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def zr():
    import __graft_entry__
    __graft_entry__.build()
    from prompt_deduplicated_shared_gb300 import zr as mod
    return mod


def test_exports_every_declared_symbol(zr):
    names = _declared_functions()
    assert len(names) >= 14
    lib = zr.lib()
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_options(zr):
    lib = zr.lib()
    assert lib.zr_version() == 100
    assert lib.zr_set_option(b"no_such_option", 1) == zr.ZR_ERR_INVALID_ARG
    assert b"unknown option" in lib.zr_last_error()
    # the dtype alone selects the attention kernels: there is no switch between them
    assert lib.zr_set_option(b"attn_impl", 0) == zr.ZR_ERR_INVALID_ARG
    assert lib.zr_set_option(b"wait_limit", -1) == zr.ZR_ERR_INVALID_ARG
    assert lib.zr_set_option(b"wait_limit", 0) == zr.ZR_OK
    assert lib.zr_set_option(b"test_withhold_arrival", 4) == zr.ZR_ERR_INVALID_ARG
    assert lib.zr_set_option(b"test_withhold_arrival", 0) == zr.ZR_OK


def test_kernel_time_without_records(zr):
    # nothing recorded yet: zero launches, no CUDA call needed
    zr.kernel_time_reset()
    assert zr.kernel_time("attn_dkdv") == (0.0, 0)
    assert zr.kernel_time("no_such_kernel") == (0.0, 0)
    lib = zr.lib()
    assert lib.zr_kernel_time(None, None, None) == zr.ZR_ERR_INVALID_ARG
    assert lib.zr_set_option(b"kernel_timing", 0) == zr.ZR_OK


def test_host_validation_without_launch(zr):
    lib = zr.lib()
    # NULL inputs
    g = zr.ZrGroupsC()
    assert lib.zr_find_prompt_groups(None, None, 4, 8, 2, ctypes.byref(g), None, None, None, 0,
                                     None) == zr.ZR_ERR_INVALID_ARG
    g = zr.ZrGroupsC(1024, 2048, 4096, 8192)  # never dereferenced on these paths
    # response_length > L
    assert lib.zr_find_prompt_groups(ctypes.c_void_p(256), None, 4, 8, 9, ctypes.byref(g), None,
                                     None, ctypes.c_void_p(256), 1 << 20, None) == zr.ZR_ERR_INVALID_ARG
    # workspace too small / misaligned
    assert lib.zr_find_prompt_groups(ctypes.c_void_p(256), None, 4, 8, 2, ctypes.byref(g), None,
                                     None, ctypes.c_void_p(256), 8, None) == zr.ZR_ERR_WORKSPACE
    assert lib.zr_find_prompt_groups(ctypes.c_void_p(256), None, 4, 8, 2, ctypes.byref(g), None,
                                     None, ctypes.c_void_p(260), 1 << 20, None) == zr.ZR_ERR_WORKSPACE
    # too many rows
    assert lib.zr_find_prompt_groups(ctypes.c_void_p(256), None, 9000, 8, 2, ctypes.byref(g), None,
                                     None, ctypes.c_void_p(256), 1 << 30, None) == zr.ZR_ERR_UNSUPPORTED
    # recon info binding
    info = zr.ZrReconInfoC()
    assert lib.zr_recon_info_bind(ctypes.byref(info), None, 4, 8, 2, 0, 32) == zr.ZR_ERR_INVALID_ARG
    assert lib.zr_recon_info_bind(ctypes.byref(info), ctypes.c_void_p(4096), 4, 8, 2, 0,
                                  33) == zr.ZR_ERR_INVALID_ARG  # T_cap > B*L
    assert lib.zr_recon_info_bind(ctypes.byref(info), ctypes.c_void_p(4096), 4, 8, 2, 0, 32) == zr.ZR_OK
    assert info.B == 4 and info.L == 8 and info.P == 6 and info.T_cap == 32
    size = lib.zr_recon_info_bytes(4)
    ptrs = [getattr(info, f) for f, _ in zr.ZrReconInfoC._fields_[:17]]
    assert all(4096 <= p < 4096 + size and p % 256 == 0 for p in ptrs)
    assert len(set(ptrs)) == 17
    # attention argument checks
    ws_bytes = lib.zr_split_attn_workspace(ctypes.byref(info), 16, 8, 128)
    assert ws_bytes > 0
    args = [ctypes.c_void_p(256)] * 5
    assert lib.zr_split_attn_fwd(ctypes.byref(info), *args, 16, 6, 128, zr.ZR_BF16, 0.0,
                                 ctypes.c_void_p(1 << 20), ws_bytes, None) == zr.ZR_ERR_UNSUPPORTED
    assert lib.zr_split_attn_fwd(ctypes.byref(info), *args, 16, 8, 80, zr.ZR_BF16, 0.0,
                                 ctypes.c_void_p(1 << 20), ws_bytes, None) == zr.ZR_ERR_UNSUPPORTED
    # bf16 head dims without a tensor-core kernel are refused, not run elsewhere
    for D in (32, 96):
        ws_d = lib.zr_split_attn_workspace(ctypes.byref(info), 16, 8, D)
        assert lib.zr_split_attn_fwd(ctypes.byref(info), *args, 16, 8, D, zr.ZR_BF16, 0.0,
                                     ctypes.c_void_p(1 << 20), ws_d, None) == zr.ZR_ERR_UNSUPPORTED
        assert b"tensor-core" in lib.zr_last_error()
    assert lib.zr_split_attn_fwd(ctypes.byref(info), *args, 16, 8, 256, zr.ZR_F32, 0.0,
                                 ctypes.c_void_p(1 << 20), ws_bytes, None) == zr.ZR_ERR_UNSUPPORTED
    assert lib.zr_split_attn_fwd(ctypes.byref(info), *args, 16, 8, 128, zr.ZR_BF16, 0.0,
                                 ctypes.c_void_p(1 << 20), ws_bytes - 1, None) == zr.ZR_ERR_WORKSPACE
    assert lib.zr_split_attn_fwd(ctypes.byref(info), None, *args[1:], 16, 8, 128, zr.ZR_BF16, 0.0,
                                 ctypes.c_void_p(1 << 20), ws_bytes, None) == zr.ZR_ERR_INVALID_ARG
    assert lib.zr_pack_rows(ctypes.byref(info), None, 8, ctypes.c_void_p(256), None) == zr.ZR_ERR_INVALID_ARG
    # batch statistics: argument checks before any launch
    bs = zr.ZrBatchStatsC()
    assert lib.zr_batch_stats_compute(None, 4, 8, 9, ctypes.byref(bs), None, 0, None) == zr.ZR_ERR_INVALID_ARG
    assert lib.zr_batch_stats_compute(None, 4, 8, 2, ctypes.byref(bs), ctypes.c_void_p(256), 8,
                                      None) == zr.ZR_ERR_WORKSPACE
    # reconstruction adjoint: element type checked before any launch
    assert lib.zr_reconstruct_backward(ctypes.byref(info), ctypes.c_void_p(256), 8, 7, ctypes.c_void_p(256),
                                       None) == zr.ZR_ERR_UNSUPPORTED
    unbound = zr.ZrReconInfoC()
    assert lib.zr_reconstruct(ctypes.byref(unbound), ctypes.c_void_p(256), 8, ctypes.c_void_p(256),
                              None) == zr.ZR_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors(zr):
    import torch
    with pytest.raises(ValueError, match="CUDA tensors only"):
        zr.find_prompt_groups(torch.zeros((2, 4), dtype=torch.int64), 1)


def test_missing_library_fails_loudly(tmp_path):
    """The binding has no fallback: without the compiled library it raises."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("from prompt_deduplicated_shared_gb300 import zr\n"
            "try:\n    zr.lib()\nexcept ImportError as e:\n    print('IMPORT_ERROR', e)\n")
    env = dict(os.environ, ZR_LIBRARY=str(tmp_path / "missing" / "libzr.so"))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert "IMPORT_ERROR" in r.stdout


def test_product_code_never_touches_the_oracle():
    """The package (binding, build script, CUDA sources) names no oracle module."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    pkg = os.path.join(root, "prompt_deduplicated_shared_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"\b(import|from)\s+oracle\b", text), f
                assert "oracle/" not in text, f
