"""GPU parity of the d = 256 forward (one Q tile per CTA, two S buffers and O
in tensor memory) through the C ABI against the fp64 oracle: dense, causal,
windowed with sink keys, varlen, strided (BHSD) and with logit sinks."""
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


def _run(ea, x, sink=None):
    o, lse = ea.attn_fwd_ex(x.q.cuda(), x.k.cuda(), x.v.cuda(), causal=x.causal, window=x.window,
                            n_sink=x.n_sink, scale=x.scale) if sink is None else \
        ea.attn_fwd_ex_sink(x.q.cuda(), x.k.cuda(), x.v.cuda(), sink_logit=sink.cuda(),
                            causal=x.causal, window=x.window, n_sink=x.n_sink, scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    return o, lse


def _check(ea, x, rows=None, sink=None, what="", stress=False):
    o, lse = _run(ea, x, sink)
    ro, rl = oracle.attn_fwd(np64(x.q), np64(x.k), np64(x.v), x.scale, x.causal, x.window,
                             x.n_sink, rows=rows,
                             sink=None if sink is None else sink.double().numpy())
    if rows is not None:
        idx = torch.as_tensor(rows, dtype=torch.long, device=o.device)
        o = o.index_select(1, idx)
        lse = lse.index_select(2, idx)
    err = compare(o, lse, ro, rl, what, stress=stress)
    masked = np.isneginf(rl).transpose(0, 2, 1)
    if masked.any() and sink is None:
        assert_masked_rows_zero(o, masked, what)
    return err


CASES = [
    # (seed, B, Hq, Hkv, Sq, Skv, causal, window, n_sink, q_mult)
    (201, 1, 1, 1, 128, 128, False, 0, 0, 1.0),      # one tile
    (202, 2, 4, 2, 300, 389, False, 0, 0, 1.0),      # ragged, several tiles, GQA
    (203, 1, 2, 2, 640, 640, True, 0, 0, 1.0),       # causal, five tiles
    (204, 1, 2, 2, 333, 333, True, 0, 0, 1.0),       # ragged causal
    (205, 1, 2, 2, 200, 700, True, 0, 0, 1.0),       # Sq < Skv: shifted diagonal
    (206, 1, 2, 2, 500, 300, True, 0, 0, 1.0),       # Sq > Skv: fully masked rows
    (207, 1, 2, 2, 512, 512, False, 0, 0, 8.0),      # scores x8: rescaling of O
    (208, 1, 2, 2, 512, 512, True, 0, 0, 8.0),       # the same, causal
    (209, 1, 2, 2, 1100, 1100, True, 128, 3, 1.0),   # narrow window, three sink keys
    (210, 1, 2, 2, 700, 1000, True, 64, 200, 1.0),   # sinks spanning tiles, Sq < Skv
    (211, 1, 4, 1, 300, 300, True, 0, 0, 1.0),       # MQA
    (212, 1, 2, 2, 1, 1, True, 0, 0, 1.0),           # single query, single key
    (213, 1, 2, 2, 129, 1, True, 0, 0, 1.0),         # one key, most rows masked
]


@pytest.mark.parametrize("case", CASES, ids=[f"seed{c[0]}" for c in CASES])
def test_small_shapes(ea, case):
    seed, B, Hq, Hkv, Sq, Skv, causal, window, n_sink, qm = case
    x = workloads.dense_inputs(seed, B, Hq, Hkv, Sq, Skv, 256, causal, window, n_sink, q_mult=qm)
    _check(ea, x, what=f"d256 seed {seed}", stress=qm != 1.0)


def test_no_keys_and_no_queries(ea):
    x = workloads.dense_inputs(214, 2, 2, 2, 70, 0, 256)
    o, lse = _run(ea, x)
    assert torch.all(o.view(torch.int16) == 0)
    assert torch.all(torch.isneginf(lse))
    x = workloads.dense_inputs(215, 1, 2, 2, 0, 64, 256)
    o, lse = _run(ea, x)
    assert o.numel() == 0


def test_deterministic(ea):
    x = workloads.dense_inputs(216, 1, 4, 2, 900, 900, 256, True)
    o1, l1 = _run(ea, x)
    o2, l2 = _run(ea, x)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


@pytest.mark.parametrize("lq,lk,causal,window,n_sink", [
    ([1, 130, 257, 600, 77], None, True, 0, 0),
    ([300, 5, 129], [100, 50, 129], True, 0, 0),     # q longer than kv: masked rows
    ([200, 513, 64], [200, 300, 1], False, 0, 0),
    ([900, 333], None, True, 100, 2),
])
def test_varlen(ea, lq, lk, causal, window, n_sink):
    x = workloads.varlen_inputs(217, len(lq), 0, 0, 8, 2, 256, causal, window, n_sink,
                                lengths=lq, klengths=lk)
    o, lse = ea.attn_fwd_ex(x.q.cuda(), x.k.cuda(), x.v.cuda(), x.cu_q.cuda(), x.cu_k.cuda(),
                            max_seqlen_q=x.max_q, max_seqlen_k=x.max_k, causal=causal,
                            window=window, n_sink=n_sink, scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    ro, rl = oracle.attn_fwd_varlen(np64(x.q), np64(x.k), np64(x.v), x.cu_q.numpy(),
                                    x.cu_k.numpy(), x.scale, causal, window, n_sink)
    compare(o, lse, ro, rl, "d256 varlen")
    masked = np.isneginf(rl).T
    if masked.any():
        assert_masked_rows_zero(o, masked, "d256 varlen")


def test_bhsd_strided(ea):
    """Q, K, V and O stored BHSD (head-major), through attn_fwd_strided; equal
    bit for bit to the contiguous call."""
    x = workloads.dense_inputs(218, 2, 4, 2, 300, 389, 256, True)
    q, k, v = (t.cuda().transpose(1, 2).contiguous().transpose(1, 2) for t in (x.q, x.k, x.v))
    o = torch.empty_like(x.q.cuda()).transpose(1, 2).contiguous().transpose(1, 2)
    o, lse = ea.attn_fwd_strided(q, k, v, o, causal=True, scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    ro, rl = oracle.attn_fwd(np64(x.q), np64(x.k), np64(x.v), x.scale, True)
    compare(o, lse, ro, rl, "d256 bhsd")
    oc, lc = _run(ea, x)
    assert torch.equal(o.contiguous().view(torch.int16), oc.view(torch.int16))
    assert torch.equal(lse, lc)


def test_logit_sinks(ea):
    x = workloads.dense_inputs(219, 1, 4, 2, 500, 300, 256, True)
    sink = workloads.logit_sinks(219, 4, lo=0.0, hi=8.0, extremes=True)
    _check(ea, x, sink=sink, what="d256 sinks")


PAGED = [
    # (seed, Hq, Hkv, key counts, query counts, causal, window, n_sink)
    (220, 4, 2, [300, 17, 1000, 129], [300, 17, 256, 1], True, 0, 0),   # prefill + decode rows
    (223, 4, 4, [100, 40, 513], [160, 40, 300], True, 0, 0),            # Lq > Lk: masked rows
    (224, 4, 2, [1500, 300], [400, 300], True, 200, 2),                 # window + sink keys
    (225, 8, 2, [600, 90], [130, 7], False, 0, 0),                      # non-causal
]


@pytest.mark.parametrize("case", PAGED, ids=[f"seed{c[0]}" for c in PAGED])
def test_paged_prefill(ea, case):
    """Query blocks against a paged cache at d = 256 (attn_fwd_paged), against
    the oracle on the same keys laid out contiguously."""
    seed, Hq, Hkv, lk, lq, causal, window, n_sink = case
    x = workloads.paged_prefill_inputs(seed, len(lk), Hq, Hkv, 256, 0, 0, 0, 0, lengths_k=lk,
                                       lengths_q=lq)
    c = x.cache
    o, lse = ea.attn_fwd_paged(x.q.cuda(), c.k_pages.cuda(), c.v_pages.cuda(),
                               c.page_table.cuda(), x.cu_q.cuda(), c.seqlens.cuda(),
                               max_seqlen_q=x.max_q, causal=causal, window=window, n_sink=n_sink,
                               scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    ro, rl = oracle.attn_fwd_varlen(np64(x.q), np64(c.k_flat), np64(c.v_flat), x.cu_q.numpy(),
                                    c.cu_kv.to(torch.int32).numpy(), x.scale, causal, window,
                                    n_sink)
    compare(o, lse, ro, rl, f"d256 paged prefill seed {seed}")
    masked = np.isneginf(rl).T
    if masked.any():
        assert_masked_rows_zero(o, masked, "d256 paged prefill")


def test_paged_prefill_bad_page_index(ea):
    """A page index outside the pool is reported and never read."""
    x = workloads.paged_prefill_inputs(226, 2, 4, 2, 256, 0, 0, 0, 0, lengths_k=[200, 64],
                                       lengths_q=[64, 64])
    c = x.cache
    pt = c.page_table.clone()
    pt[0, 2] = c.k_pages.shape[0] + 5
    ea.attn_fwd_paged(x.q.cuda(), c.k_pages.cuda(), c.v_pages.cuda(), pt.cuda(), x.cu_q.cuda(),
                      c.seqlens.cuda(), max_seqlen_q=x.max_q, causal=True, scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_ERR_BAD_INPUT
    assert ea.attn_device_status() == ea.ATTN_OK


@pytest.mark.parametrize("Hq,Hkv,splits", [(8, 2, 1), (8, 2, 3), (32, 8, 8), (4, 4, 5),
                                           (64, 2, 4)])
def test_decode(ea, Hq, Hkv, splits):
    """Paged split-KV decode at d = 256 against the oracle (empty, one-token,
    page-boundary and long requests; more splits than pages)."""
    lengths = [1, 15, 16, 17, 300, 0, 64, 1000]
    x = workloads.paged_decode_inputs(227, len(lengths), Hq, Hkv, 256, 0, 0, lengths=lengths,
                                      num_splits=splits, extra_pages=7)
    o, lse = ea.attn_decode_paged(x.q.cuda(), x.k_pages.cuda(), x.v_pages.cuda(),
                                  x.page_table.cuda(), x.seqlens.cuda(), num_splits=splits,
                                  scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    k, v = x.contiguous_kv(list(range(len(lengths))))
    ro, rl = oracle.attn_decode(np64(x.q), np64(k), np64(v), x.seqlens.numpy(), x.scale)
    compare(o, lse, ro, rl, f"d256 decode Hq={Hq} Hkv={Hkv} S={splits}")
    assert_masked_rows_zero(o, np.isneginf(rl), "d256 decode empty request")


def test_decode_batch(ea):
    """B=16 requests of 1024-8192 keys, Hq=32, Hkv=8, 8 splits, d = 256, with
    logit sinks too; every request against the oracle."""
    x = workloads.paged_decode_inputs(228, 16, 32, 8, 256, 1024, 8192, num_splits=8)
    q, kp, vp, pt, sl = (t.cuda() for t in (x.q, x.k_pages, x.v_pages, x.page_table, x.seqlens))
    o, lse = ea.attn_decode_paged(q, kp, vp, pt, sl, num_splits=8, scale=x.scale)
    sink = workloads.logit_sinks(228, 32)
    os_, ls_ = ea.attn_decode_paged_sink(q, kp, vp, pt, sl, sink.cuda(), num_splits=8,
                                         scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    for c in range(0, 16, 4):
        req = list(range(c, c + 4))
        k, v = x.contiguous_kv(req)
        ro, rl = oracle.attn_decode(np64(x.q[req]), np64(k), np64(v), x.seqlens[req].numpy(),
                                    x.scale)
        compare(o[c:c + 4], lse[c:c + 4], ro, rl, f"d256 decode requests {c}..{c + 3}")
        ro, rl = oracle.attn_decode(np64(x.q[req]), np64(k), np64(v), x.seqlens[req].numpy(),
                                    x.scale, sink=sink.double().numpy())
        compare(os_[c:c + 4], ls_[c:c + 4], ro, rl, f"d256 decode sinks {c}..{c + 3}")


@pytest.mark.parametrize("causal", [False, True])
def test_full_size_sampled(ea, causal):
    """B=4, H=16, S=2048, d=256 (the size bench.py times): sampled rows of
    every (batch, head) against the oracle."""
    x = workloads.dense_inputs(221 + int(causal), 4, 16, 16, 2048, 2048, 256, causal)
    err = _check(ea, x, rows=sample_rows(2048), what=f"d256 full c={causal}")
    print(f"d256 full causal={causal}: max |dO| {err[0]:.2e}, max |dLSE| {err[1]:.2e}, "
          f"{err[2]} elements with |O| >= 4")


def test_persistent_items_without_keys(ea):
    """More Q tiles than SMs with Sq > Skv (causal): the persistent grid's CTAs
    walk items whose rows see no key (O = 0, LSE = -inf) between ones that
    do; sampled rows against the oracle, the masked rows checked bit for bit."""
    x = workloads.dense_inputs(229, 2, 16, 8, 1200, 600, 256, True)
    rows = sample_rows(1200, seed=229)
    _check(ea, x, rows=rows, what="d256 persistent, rows without keys")
