"""The C-ABI library builds, loads and exports every entry point that
include/attn.h declares; argument checks that run before any CUDA call
answer without a GPU.  No compute call is made here."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("attn_fwd", "attn_fwd_ex", "attn_decode_paged", "attn_decode_workspace_size",
              "attn_device_status", "attn_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol():
    import exact_attention_08_gb300 as ea
    out = subprocess.run(["nm", "-D", "--defined-only", ea.library_path], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(attn_\w+)", out))
    missing = set(declared_symbols()) - exported
    assert not missing, f"not exported: {missing}"
    # nothing but the declared ABI leaks out
    assert exported == set(declared_symbols())


def test_status_strings():
    import exact_attention_08_gb300 as ea
    for code in range(6):
        assert ea.attn_status_string(code) != "unknown status"
    assert ea.attn_status_string(99) == "unknown status"


def test_argument_errors_without_gpu():
    import exact_attention_08_gb300 as ea
    L = ea.lib
    buf = ctypes.create_string_buffer(64)
    p = ctypes.cast(buf, ctypes.c_void_p).value
    p16 = (p + 15) & ~15
    # Hq not a multiple of Hkv
    assert L.attn_fwd(p16, p16, p16, p16, None, 1, 3, 2, 8, 8, 128, 0.1, 0, 0, None) == ea.ATTN_ERR_INVALID_ARG
    # unsupported head dim
    assert L.attn_fwd(p16, p16, p16, p16, None, 1, 2, 2, 8, 8, 96, 0.1, 0, 0, None) == ea.ATTN_ERR_UNSUPPORTED
    # window without causal; sinks without window; non-positive scale
    assert L.attn_fwd(p16, p16, p16, p16, None, 1, 2, 2, 8, 8, 128, 0.1, 0, 4, None) == ea.ATTN_ERR_INVALID_ARG
    assert L.attn_fwd_ex(p16, p16, p16, p16, None, None, None, 1, 2, 2, 8, 8, 0, 0, 128, 0.1, 1, 0,
                         1, None) == ea.ATTN_ERR_INVALID_ARG
    assert L.attn_fwd(p16, p16, p16, p16, None, 1, 2, 2, 8, 8, 128, -1.0, 0, 0, None) == ea.ATTN_ERR_INVALID_ARG
    # misaligned pointer
    assert L.attn_fwd(p16 + 2, p16, p16, p16, None, 1, 2, 2, 8, 8, 128, 0.1, 0, 0, None) == ea.ATTN_ERR_INVALID_ARG
    # one cu_seqlens without the other
    assert L.attn_fwd_ex(p16, p16, p16, p16, None, p16, None, 1, 2, 2, 8, 8, 8, 8, 128, 0.1, 1, 0,
                         0, None) == ea.ATTN_ERR_INVALID_ARG
    # empty problem: nothing to launch
    assert L.attn_fwd(None, None, None, None, None, 0, 2, 2, 8, 8, 128, 0.1, 0, 0, None) == ea.ATTN_OK
    assert L.attn_fwd(None, None, None, None, None, 2, 2, 2, 0, 8, 128, 0.1, 0, 0, None) == ea.ATTN_OK
    assert "multiple" in ea.attn_last_error() or ea.attn_last_error() == ""


def test_decode_argument_errors_without_gpu():
    import exact_attention_08_gb300 as ea
    L = ea.lib
    buf = ctypes.create_string_buffer(64)
    p16 = (ctypes.cast(buf, ctypes.c_void_p).value + 15) & ~15
    # split outputs and log-sum-exps (fp32), the request order (int32)
    assert L.attn_decode_workspace_size(64, 32, 128, 8) == 64 * 32 * 8 * (128 + 1) * 4 + 64 * 4
    assert L.attn_decode_workspace_size(-1, 32, 128, 8) == 0
    args = [p16, p16, p16, p16, p16, p16, None, 2, 8, 2, 128, 16, 4, 10, 8, 0.1, p16, 1 << 20, None]
    bad = list(args)
    bad[11] = 32  # page size
    assert L.attn_decode_paged(*bad) == ea.ATTN_ERR_UNSUPPORTED
    bad = list(args)
    bad[14] = 0   # num_splits
    assert L.attn_decode_paged(*bad) == ea.ATTN_ERR_INVALID_ARG
    bad = list(args)
    bad[17] = 16  # workspace too small
    assert L.attn_decode_paged(*bad) == ea.ATTN_ERR_INVALID_ARG
    bad = list(args)
    bad[8] = 3    # Hq % Hkv
    assert L.attn_decode_paged(*bad) == ea.ATTN_ERR_INVALID_ARG
    assert L.attn_check_wait_timeout(0, None) == ea.ATTN_ERR_INVALID_ARG


def test_argument_errors_of_the_newer_entry_points_without_gpu():
    """Checks that run before any CUDA call: the strided, paged, sink and
    backward entry points reject bad arguments without a device."""
    import exact_attention_08_gb300 as ea
    L = ea.lib
    buf = ctypes.create_string_buffer(256)
    p = ctypes.cast(buf, ctypes.c_void_p).value
    p16 = (p + 15) & ~15
    S3 = ctypes.c_longlong * 3
    # strided: a stride that is not a multiple of 16 bytes
    bad = S3(128 * 2 * 64, 128 * 2 + 4, 128)
    assert L.attn_fwd_strided(p16, p16, p16, p16, None, 1, 2, 2, 64, 64, 128, bad, None, None,
                              None, 0.1, 0, 0, 0, None, None) == ea.ATTN_ERR_INVALID_ARG
    # paged: page size other than 16, head dim 96, window without causal
    assert L.attn_fwd_paged(p16, p16, p16, p16, p16, p16, p16, None, 1, 2, 2, 8, 8, 128, 32, 4,
                            4, 0.1, 1, 0, 0, None, None) == ea.ATTN_ERR_UNSUPPORTED
    assert L.attn_fwd_paged(p16, p16, p16, p16, p16, p16, p16, None, 1, 2, 2, 8, 8, 96, 16, 4,
                            4, 0.1, 1, 0, 0, None, None) == ea.ATTN_ERR_UNSUPPORTED
    assert L.attn_fwd_paged(p16, p16, p16, p16, p16, p16, p16, None, 1, 2, 2, 8, 8, 128, 16, 4,
                            4, 0.1, 0, 8, 0, None, None) == ea.ATTN_ERR_INVALID_ARG
    # sink: a misaligned sink pointer
    assert L.attn_fwd_ex_sink(p16, p16, p16, p16, None, None, None, 1, 2, 2, 8, 8, 0, 0, 128, 0.1,
                              0, 0, 0, p16 + 2, None) == ea.ATTN_ERR_INVALID_ARG
    # backward: Hq not a multiple of Hkv, too small a workspace
    assert L.attn_bwd(p16, p16, p16, p16, p16, p16, p16, p16, p16, 1, 3, 2, 8, 8, 128, 0.1, 0,
                      p16, 1 << 20, None) == ea.ATTN_ERR_INVALID_ARG
    assert L.attn_bwd(p16, p16, p16, p16, p16, p16, p16, p16, p16, 1, 2, 2, 300, 8, 128, 0.1, 0,
                      p16, 16, None) == ea.ATTN_ERR_INVALID_ARG
    assert ea.attn_bwd_workspace_size(1, 2, 300) == 2 * 2 * 384 * 4
    # d = 64, 128 and 256 run in every call; other head dimensions are
    # rejected before any launch
    assert L.attn_bwd(p16, p16, p16, p16, p16, p16, p16, p16, p16, 1, 2, 2, 8, 8, 192, 0.1, 0,
                      p16, 1 << 20, None) == ea.ATTN_ERR_UNSUPPORTED
    assert "192" in ea.attn_last_error()
    assert L.attn_fwd_paged(p16, p16, p16, p16, p16, p16, p16, None, 1, 2, 2, 8, 8, 96, 16, 4,
                            4, 0.1, 1, 0, 0, None, None) == ea.ATTN_ERR_UNSUPPORTED
    assert L.attn_decode_paged(p16, p16, p16, p16, p16, p16, None, 2, 8, 2, 192, 16, 4, 10, 8, 0.1,
                               p16, 1 << 20, None) == ea.ATTN_ERR_UNSUPPORTED
    assert "192" in ea.attn_last_error()


def test_backward_sink_argument_errors_without_gpu():
    """attn_bwd_ex_sink wants both sink pointers, 4-byte aligned; both checks
    answer before any CUDA call."""
    import exact_attention_08_gb300 as ea
    L = ea.lib
    buf = ctypes.create_string_buffer(256)
    p = ctypes.cast(buf, ctypes.c_void_p).value
    p16 = (p + 15) & ~15
    args = (p16, p16, p16, p16, p16, p16, p16, p16, p16, None, None, 1, 2, 2, 8, 8, 0, 0, 128,
            0.1, 0, 0, 0)
    tail = (p16, 1 << 20, None)
    assert L.attn_bwd_ex_sink(*args, p16, None, *tail) == ea.ATTN_ERR_INVALID_ARG
    assert L.attn_bwd_ex_sink(*args, None, p16, *tail) == ea.ATTN_ERR_INVALID_ARG
    assert L.attn_bwd_ex_sink(*args, p16 + 2, p16, *tail) == ea.ATTN_ERR_INVALID_ARG
    assert "sink" in ea.attn_last_error()
