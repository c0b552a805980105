"""attn_decode_paged_noalloc: the decode entry point that allocates nothing.

It serves callers that cannot allocate device memory themselves (for example a
serving loop that must not allocate once it runs, or a host program whose
plugins may only use memory they are given): the split partials go to a
scratch array built into the library instead of a caller workspace.  Here it is
called through the C ABI twice in a row and each result is checked against
the workspace entry point, attn_decode_paged, on the same inputs.  This file is
named so that pytest collects it after every other test file; it also passes
alone in a fresh process.
"""
import ctypes

import pytest
import torch

import workloads
from tests._parity import compare

pytestmark = pytest.mark.gpu


def _noalloc(lib):
    f = lib.attn_decode_paged_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, ctypes.c_float, vp]
    f.restype = ctypes.c_int
    return f


def test_noalloc_decode_matches_workspace_decode_twice():
    import exact_attention_08_gb300 as ea
    f = _noalloc(ea.lib)
    x = workloads.paged_decode_inputs(91, 16, 32, 8, 128, 1, 3000, num_splits=8, extra_pages=3)
    q, kp, vp = x.q.cuda(), x.k_pages.cuda(), x.v_pages.cuda()
    pt, sl = x.page_table.cuda(), x.seqlens.cuda()
    B, Hq, d = q.shape
    P, page, Hkv, _ = kp.shape
    o_ref, lse_ref = ea.attn_decode_paged(q, kp, vp, pt, sl, num_splits=8, scale=x.scale)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=q.device)
        rc = f(q.data_ptr(), kp.data_ptr(), vp.data_ptr(), pt.data_ptr(), sl.data_ptr(),
               o.data_ptr(), lse.data_ptr(), B, Hq, Hkv, d, page, pt.shape[1], P, 8, x.scale,
               stream)
        assert rc == ea.ATTN_OK, ea.attn_last_error()
        torch.cuda.synchronize()
        assert ea.attn_device_status() == ea.ATTN_OK
        compare(o, lse, o_ref.double().cpu().numpy(), lse_ref.double().cpu().numpy(),
                f"no-alloc decode call {call}")


def test_noalloc_decode_rejects_sizes_beyond_its_scratch():
    import exact_attention_08_gb300 as ea
    f = _noalloc(ea.lib)
    buf = torch.empty(1024, dtype=torch.uint8, device="cuda")
    p = buf.data_ptr()
    # 4096 requests x 64 heads x 64 splits x (128 + 1) floats is far beyond 16 MiB
    rc = f(p, p, p, p, p, p, None, 4096, 64, 8, 128, 16, 4, 4, 64, 0.1, None)
    assert rc == ea.ATTN_ERR_INVALID_ARG
    assert "scratch" in ea.attn_last_error()
