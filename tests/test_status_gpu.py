"""Failure reporting on the GPU without faulting it: a bounded wait that runs
out sets the device status word, the kernel returns, and the context stays
usable for the next call."""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


def test_bounded_wait_timeout_reported_and_context_usable():
    import exact_attention_08_gb300 as ea
    assert ea.attn_device_status() == ea.ATTN_OK
    ea.attn_check_wait_timeout(2000)  # 2 ms on a barrier nothing completes
    assert ea.attn_device_status() == ea.ATTN_ERR_TIMEOUT
    assert ea.attn_device_status() == ea.ATTN_OK
    x = workloads.dense_inputs(61, 1, 2, 2, 256, 256, 128, causal=True)
    o, lse = ea.attn_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), causal=True)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    assert torch.isfinite(o.float()).all()


def test_argument_errors_launch_nothing():
    import exact_attention_08_gb300 as ea
    x = workloads.dense_inputs(62, 1, 3, 2, 64, 64, 128)
    with pytest.raises(ea.AttnError) as e:
        ea.attn_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda())  # Hq=3 not a multiple of Hkv=2
    assert e.value.status == ea.ATTN_ERR_INVALID_ARG
    x = workloads.dense_inputs(63, 1, 2, 2, 64, 64, 96)
    with pytest.raises(ea.AttnError) as e:
        ea.attn_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda())
    assert e.value.status == ea.ATTN_ERR_UNSUPPORTED
    x = workloads.dense_inputs(64, 1, 2, 2, 64, 64, 128)
    with pytest.raises(ea.AttnError) as e:
        ea.attn_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), causal=False, window=16)
    assert e.value.status == ea.ATTN_ERR_INVALID_ARG
    assert ea.attn_device_status() == ea.ATTN_OK
