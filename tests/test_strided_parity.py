"""GPU parity of attn_fwd_strided (dense forward on any layout with a
contiguous head dimension: BHSD, mixed, padded) through the C ABI against
the fp64 oracle, and bit equality with the contiguous call."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._parity import compare, np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ea():
    import exact_attention_08_gb300 as m
    assert torch.cuda.is_available()
    return m


def _bhsd_view(t):
    """The same values stored BHSD, viewed in BSHD index order."""
    return t.transpose(1, 2).contiguous().transpose(1, 2)


def _padded_view(t, pad):
    """BSHD index order with `pad` extra elements after every head row."""
    B, S, H, d = t.shape
    buf = torch.full((B, S, H, d + pad), 7.0, dtype=t.dtype, device=t.device)
    buf[..., :d] = t
    return buf[..., :d]


CASES = [
    # (seed, B, Hq, Hkv, Sq, Skv, d, causal, window, n_sink)
    (91, 2, 4, 2, 300, 389, 128, False, 0, 0),
    (92, 1, 4, 4, 640, 640, 128, True, 0, 0),
    (93, 2, 8, 2, 257, 513, 64, True, 0, 0),
    (94, 1, 2, 2, 1100, 1100, 128, True, 128, 3),
]


@pytest.mark.parametrize("case", CASES, ids=[f"seed{c[0]}" for c in CASES])
@pytest.mark.parametrize("layout", ["bhsd", "mixed", "padded"])
def test_layouts(ea, case, layout):
    seed, B, Hq, Hkv, Sq, Skv, d, causal, window, n_sink = case
    x = workloads.dense_inputs(seed, B, Hq, Hkv, Sq, Skv, d, causal, window, n_sink)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    if layout == "bhsd":
        qs, ks, vs = _bhsd_view(q), _bhsd_view(k), _bhsd_view(v)
        o = None
    elif layout == "mixed":
        qs, ks, vs = q, _bhsd_view(k), _bhsd_view(v)
        o = _bhsd_view(torch.empty_like(q))
    else:
        qs, ks, vs = _padded_view(q, 64), _padded_view(k, 8), _padded_view(v, 128)
        o = _padded_view(torch.empty_like(q), 32)
    o, lse = ea.attn_fwd_strided(qs, ks, vs, o, causal=causal, window=window, n_sink=n_sink,
                                 scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    ro, rl = oracle.attn_fwd(np64(x.q), np64(x.k), np64(x.v), x.scale, causal, window, n_sink)
    compare(o, lse, ro, rl, f"{layout} seed {seed}")
    oc, lc = ea.attn_fwd_ex(q, k, v, causal=causal, window=window, n_sink=n_sink, scale=x.scale)
    torch.cuda.synchronize()
    assert torch.equal(o.contiguous().view(torch.int16), oc.view(torch.int16))
    assert torch.equal(lse, lc)
    if layout == "padded":  # the padding after each row is untouched
        base = o.as_strided((B, Sq, Hq, d + 32), (o.stride(0), o.stride(1), o.stride(2), 1))
        assert torch.all(base[..., d:] == 7.0)


def test_sink_logits_bhsd(ea):
    x = workloads.dense_inputs(95, 1, 4, 2, 500, 300, 128, True)
    sink = workloads.logit_sinks(95, 4, lo=0.0, hi=8.0, extremes=True).cuda()
    q, k, v = (_bhsd_view(t.cuda()) for t in (x.q, x.k, x.v))
    o, lse = ea.attn_fwd_strided(q, k, v, causal=True, sink_logit=sink, scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    ro, rl = oracle.attn_fwd(np64(x.q), np64(x.k), np64(x.v), x.scale, True,
                             sink=sink.double().cpu().numpy())
    compare(o, lse, ro, rl, "bhsd with sinks")


def test_no_keys_fills_strided_output(ea):
    """Skv = 0: O = 0 at the strided positions only, LSE = -inf."""
    x = workloads.dense_inputs(96, 2, 4, 4, 70, 0, 128)
    q = _bhsd_view(x.q.cuda())
    k = v = torch.empty(2, 0, 4, 128, dtype=torch.bfloat16, device="cuda")
    o = _padded_view(torch.empty_like(x.q.cuda()), 64)
    o, lse = ea.attn_fwd_strided(q, k, v, o, scale=x.scale)
    torch.cuda.synchronize()
    assert torch.all(o.view(torch.int16) == 0)
    base = o.as_strided((2, 70, 4, 192), (o.stride(0), o.stride(1), o.stride(2), 1))
    assert torch.all(base[..., 128:] == 7.0)
    assert torch.all(torch.isneginf(lse))


def test_bad_stride_is_rejected(ea):
    x = workloads.dense_inputs(97, 1, 2, 2, 64, 64, 128)
    q = _padded_view(x.q.cuda(), 4)  # head stride 132 elements: not a multiple of 16 bytes
    with pytest.raises(ea.AttnError) as e:
        ea.attn_fwd_strided(q, x.k.cuda(), x.v.cuda(), scale=x.scale)
    assert e.value.status == ea.ATTN_ERR_INVALID_ARG
