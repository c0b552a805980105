"""GPU parity of attn_fwd_paged (packed query blocks against a paged KV cache,
through the C ABI) against the fp64 oracle on the same keys laid out
contiguously ("TileLang tutorial, ch.15", sections 3.4(2) and 5.3: causal
alignment to the end of each sequence's keys)."""
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


def _run(ea, x, causal=True, window=0, n_sink=0, sink=None, page_table=None):
    c = x.cache
    pt = (c.page_table if page_table is None else page_table).cuda()
    o, lse = ea.attn_fwd_paged(x.q.cuda(), c.k_pages.cuda(), c.v_pages.cuda(), pt,
                               x.cu_q.cuda(), c.seqlens.cuda(), max_seqlen_q=x.max_q,
                               causal=causal, window=window, n_sink=n_sink,
                               sink_logit=None if sink is None else sink.cuda(), scale=x.scale)
    torch.cuda.synchronize()
    return o, lse


def _oracle(x, causal=True, window=0, n_sink=0, sink=None):
    c = x.cache
    return oracle.attn_fwd_varlen(np64(x.q), np64(c.k_flat), np64(c.v_flat), x.cu_q.numpy(),
                                  c.cu_kv.to(torch.int32).numpy(), x.scale, causal, window, n_sink,
                                  sink=None if sink is None else sink.double().numpy())


CASES = [
    # (seed, Hq, Hkv, d, key counts, query counts, causal, window, n_sink)
    (81, 4, 2, 128, [300, 17, 1000, 129], [300, 17, 256, 1], True, 0, 0),   # prefill + decode rows
    (82, 8, 2, 128, [700, 64, 2050], [4, 4, 4], True, 0, 0),                 # speculative blocks
    (83, 4, 4, 128, [100, 40, 513], [160, 40, 300], True, 0, 0),             # Lq > Lk: masked rows
    (84, 4, 1, 64, [900, 33], [129, 257], True, 0, 0),                       # d=64, MQA, ragged
    (85, 4, 2, 128, [1500, 300], [400, 300], True, 200, 2),                  # window + sink keys
    (86, 4, 2, 128, [600, 90], [130, 7], False, 0, 0),                       # non-causal
]


@pytest.mark.parametrize("case", CASES, ids=[f"seed{c[0]}" for c in CASES])
def test_small(ea, case):
    seed, Hq, Hkv, d, lk, lq, causal, window, n_sink = case
    x = workloads.paged_prefill_inputs(seed, len(lk), Hq, Hkv, d, 0, 0, 0, 0, lengths_k=lk,
                                       lengths_q=lq)
    o, lse = _run(ea, x, causal, window, n_sink)
    assert ea.attn_device_status() == ea.ATTN_OK
    ro, rl = _oracle(x, causal, window, n_sink)
    compare(o, lse, ro, rl, f"paged prefill seed {seed}")
    masked = np.isneginf(rl).T  # [Tq, Hq]
    if masked.any():
        assert_masked_rows_zero(o, masked, f"paged prefill seed {seed}")


def test_with_logit_sinks(ea):
    x = workloads.paged_prefill_inputs(87, 3, 4, 2, 128, 0, 0, 0, 0, lengths_k=[800, 20, 300],
                                       lengths_q=[200, 40, 3])
    sink = workloads.logit_sinks(87, 4, lo=0.0, hi=8.0, extremes=True)
    o, lse = _run(ea, x, sink=sink)
    assert ea.attn_device_status() == ea.ATTN_OK
    ro, rl = _oracle(x, sink=sink)
    compare(o, lse, ro, rl, "paged prefill with sinks")
    # Lq = 40 > Lk = 20: the first 20 rows of sequence 1 see no key
    rows = slice(200, 220)
    assert torch.all(o[rows].view(torch.int16) == 0)
    assert torch.equal(lse[:, rows], sink.cuda()[:, None].expand(4, 20))


def test_one_row_blocks_equal_decode(ea):
    """A block of one query row per sequence is the decode of that row."""
    x = workloads.paged_prefill_inputs(88, 5, 8, 2, 128, 0, 0, 0, 0,
                                       lengths_k=[1, 16, 17, 1000, 333], lengths_q=[1] * 5)
    o, lse = _run(ea, x)
    c = x.cache
    od, ld = ea.attn_decode_paged(x.q.cuda(), c.k_pages.cuda(), c.v_pages.cuda(),
                                  c.page_table.cuda(), c.seqlens.cuda(), num_splits=1,
                                  scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    assert (o.float() - od.float()).abs().max().item() < 2e-2
    assert (lse.T - ld).abs().max().item() < 2e-3


def test_page_index_out_of_range_is_reported(ea):
    """An entry outside the page pool is not dereferenced: page 0 is read in
    its place and the call reports ATTN_ERR_BAD_INPUT."""
    x = workloads.paged_prefill_inputs(89, 2, 4, 2, 128, 0, 0, 0, 0, lengths_k=[300, 100],
                                       lengths_q=[64, 64])
    pt = x.cache.page_table.clone()
    pt[0, 3] = x.cache.k_pages.shape[0] + 5
    o, lse = _run(ea, x, page_table=pt)
    assert ea.attn_device_status() == ea.ATTN_ERR_BAD_INPUT
    assert ea.attn_device_status() == ea.ATTN_OK  # cleared by the read


def test_chunked_prefill_full_size(ea):
    """B=8, Hq=32, Hkv=8, d=128, caches of 2048-8192 keys, 512-row query blocks:
    sampled rows of every sequence against the dense oracle of that sequence."""
    x = workloads.chunked_prefill()
    o, lse = _run(ea, x)
    assert ea.attn_device_status() == ea.ATTN_OK
    c = x.cache
    cu_q, cu_k = x.cu_q.tolist(), c.cu_kv.tolist()
    for b in range(len(cu_q) - 1):
        lq = cu_q[b + 1] - cu_q[b]
        rows = sample_rows(lq, seed=9 + b)
        qb = np64(x.q[cu_q[b]:cu_q[b + 1]])[None]
        kb = np64(c.k_flat[cu_k[b]:cu_k[b + 1]])[None]
        vb = np64(c.v_flat[cu_k[b]:cu_k[b + 1]])[None]
        ro, rl = oracle.attn_fwd(qb, kb, vb, x.scale, True, rows=rows)
        idx = torch.as_tensor(cu_q[b] + rows, dtype=torch.long, device=o.device)
        compare(o.index_select(0, idx)[None], lse.index_select(1, idx)[None], ro, rl,
                f"chunked prefill sequence {b}")


@pytest.mark.parametrize("nseq,seed", [(50, 87), (80, 88)])
def test_many_sequences(ea, nseq, seed):
    """Causal query blocks of 0-300 rows against caches of 0-1,500 keys: 50
    sequences (dealt by key count, two per lane of the ordering warp) and 80
    (past that bound: dealt by query pair), empty blocks and caches among
    them, against the oracle."""
    r = np.random.default_rng(seed)
    lk = r.integers(0, 1500, nseq).tolist()
    lq = [int(min(q, k)) for q, k in zip(r.integers(0, 300, nseq), lk)]
    x = workloads.paged_prefill_inputs(seed, nseq, 4, 2, 128, 0, 0, 0, 0, lengths_k=lk,
                                       lengths_q=lq)
    o, lse = _run(ea, x)
    assert ea.attn_device_status() == ea.ATTN_OK
    ro, rl = _oracle(x)
    compare(o, lse, ro, rl, f"paged prefill, {nseq} sequences")
