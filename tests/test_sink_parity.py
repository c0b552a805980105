"""GPU parity of the logit-sink entry points (attn_fwd_ex_sink,
attn_decode_paged_sink, through the C ABI) against the fp64 oracle with the
same per-head sinks ("TileLang tutorial, ch.15", section 4.6)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._parity import assert_masked_rows_zero, compare, np64, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ea():
    import exact_attention_08_gb300 as m
    assert torch.cuda.is_available()
    return m


def _run(ea, x, sink, stream=None):
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    o, lse = ea.attn_fwd_ex_sink(q, k, v, sink.cuda(), causal=x.causal, window=x.window,
                                 n_sink=x.n_sink, scale=x.scale, stream=stream)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    return o, lse


def _check(ea, x, sink, rows=None, what=""):
    o, lse = _run(ea, x, sink)
    ro, rl = oracle.attn_fwd(np64(x.q), np64(x.k), np64(x.v), x.scale, x.causal, x.window,
                             x.n_sink, rows=rows, sink=sink.double().numpy())
    if rows is not None:
        idx = torch.as_tensor(rows, dtype=torch.long, device=o.device)
        o = o.index_select(1, idx)
        lse = lse.index_select(2, idx)
    compare(o, lse, ro, rl, what)
    masked = np.isneginf(rl).transpose(0, 2, 1)
    if masked.any():
        assert_masked_rows_zero(o, masked, what)
    return o, lse, ro, rl


CASES = [
    # (seed, B, Hq, Hkv, Sq, Skv, d, causal, window, n_sink)
    (61, 1, 4, 4, 300, 389, 128, False, 0, 0),     # ragged, several tiles
    (62, 2, 4, 2, 333, 333, 128, True, 0, 0),      # ragged causal, GQA 2:1
    (63, 1, 4, 4, 500, 300, 128, True, 0, 0),      # Sq > Skv: rows with no key
    (64, 1, 4, 4, 1100, 1100, 128, True, 128, 3),   # window + sink keys
    (65, 1, 8, 2, 300, 300, 64, True, 0, 0),       # d=64, GQA 4:1
    (66, 1, 4, 4, 1, 1, 128, True, 0, 0),          # single query, single key
]


@pytest.mark.parametrize("case", CASES, ids=[f"seed{c[0]}" for c in CASES])
def test_small_shapes_with_sinks(ea, case):
    seed, B, Hq, Hkv, Sq, Skv, d, causal, window, n_sink = case
    x = workloads.dense_inputs(seed, B, Hq, Hkv, Sq, Skv, d, causal, window, n_sink)
    sink = workloads.logit_sinks(seed, Hq, lo=0.0, hi=8.0, extremes=True)
    o, lse, ro, rl = _check(ea, x, sink, what=f"sink case seed {seed}")
    # head 1 has a dominant sink (e^100 overflows fp32): O ~ 0, LSE = 100
    assert float(o[:, :, 1].float().abs().max()) < 1e-6
    assert torch.allclose(lse[:, 1], torch.full_like(lse[:, 1], 100.0), atol=1e-3, rtol=0)


def test_rows_without_keys_take_the_sink(ea):
    """Causal with Sq > Skv: the first rows see no key: O = +0.0 exactly and
    LSE = the head's sink (or -inf where the sink is -inf)."""
    x = workloads.dense_inputs(67, 1, 4, 4, 260, 100, 128, True)
    sink = workloads.logit_sinks(67, 4, extremes=True)
    o, lse = _run(ea, x, sink)
    n = 260 - 100
    assert torch.all(o[:, :n].view(torch.int16) == 0)
    exp = sink.cuda()[None, :, None].expand(1, 4, n)
    assert torch.equal(lse[:, :, :n], exp)


def test_no_keys_at_all(ea):
    """Skv = 0: every row gets O = 0 and LSE = its head's sink."""
    x = workloads.dense_inputs(68, 2, 4, 4, 70, 0, 128)
    sink = workloads.logit_sinks(68, 4, extremes=True)
    o, lse = _run(ea, x, sink)
    assert torch.all(o.view(torch.int16) == 0)
    assert torch.equal(lse, sink.cuda()[None, :, None].expand(2, 4, 70))


def test_minus_inf_sinks_equal_the_plain_forward(ea):
    """Sinks of -inf everywhere give the same bits as attn_fwd_ex."""
    x = workloads.dense_inputs(69, 1, 4, 2, 700, 700, 128, True)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    o1, l1 = ea.attn_fwd_ex(q, k, v, causal=True, scale=x.scale)
    o2, l2 = ea.attn_fwd_ex_sink(q, k, v, torch.full((4,), float("-inf"), device="cuda"),
                                 causal=True, scale=x.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


def test_varlen_with_sinks(ea):
    x = workloads.varlen_inputs(70, 4, 1, 700, 4, 2, 128, causal=True)
    sink = workloads.logit_sinks(70, 4, extremes=True)
    cu_q, cu_k = x.cu_q.to(torch.int32).cuda(), x.cu_k.to(torch.int32).cuda()
    o, lse = ea.attn_fwd_ex_sink(x.q.cuda(), x.k.cuda(), x.v.cuda(), sink.cuda(), cu_q, cu_k,
                                 max_seqlen_q=x.max_q, max_seqlen_k=x.max_k, causal=True,
                                 scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    ro, rl = oracle.attn_fwd_varlen(np64(x.q), np64(x.k), np64(x.v), x.cu_q.numpy(),
                                    x.cu_k.numpy(), x.scale, True, sink=sink.double().numpy())
    compare(o, lse, ro, rl, "varlen with sinks")


@pytest.mark.parametrize("causal", [False, True])
def test_prefill_full_size_with_sinks(ea, causal):
    """B=4, H=16, S=2048, d=128 with sinks in [4, 12]; sampled rows against the oracle."""
    x = workloads.prefill_mha(causal)
    sink = workloads.logit_sinks(2100 + int(causal), 16)
    _check(ea, x, sink, rows=sample_rows(2048, seed=5), what=f"full size, causal={causal}")


@pytest.mark.parametrize("num_splits,hd", [(1, 128), (8, 128), (3, 256), (8, 64)])
def test_decode_with_sinks(ea, num_splits, hd):
    d = workloads.paged_decode_inputs(71, 6, 8, 2, hd, 1, 900, num_splits=num_splits,
                                      lengths=[900, 0, 1, 17, 256, 640])
    sink = workloads.logit_sinks(71, 8, lo=0.0, hi=8.0, extremes=True)
    o, lse = ea.attn_decode_paged_sink(d.q.cuda(), d.k_pages.cuda(), d.v_pages.cuda(),
                                       d.page_table.cuda(), d.seqlens.cuda(), sink.cuda(),
                                       num_splits=num_splits, scale=d.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    req = list(range(6))
    k, v = d.contiguous_kv(req)
    ro, rl = oracle.attn_decode(np64(d.q), np64(k), np64(v), d.seqlens.numpy(), d.scale,
                                sink=sink.double().numpy())
    compare(o, lse, ro, rl, f"decode with sinks, splits={num_splits}, d={hd}")
    # request 1 has no key: O = 0, LSE = sink
    assert torch.all(o[1].view(torch.int16) == 0)
    assert torch.equal(lse[1], sink.cuda())
