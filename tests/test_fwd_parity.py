"""GPU parity of the prefill forward (attn_fwd / attn_fwd_ex through the C ABI)
against the fp64 oracle on the same seeded bf16 inputs."""
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


def run_dense(ea, x, stream=None):
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    o, lse = ea.attn_fwd_ex(q, k, v, causal=x.causal, window=x.window, n_sink=x.n_sink,
                            scale=x.scale, stream=stream)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    return o, lse


def check_dense(ea, x, rows=None, what="", stress=False):
    o, lse = run_dense(ea, x)
    ro, rl = oracle.attn_fwd(np64(x.q), np64(x.k), np64(x.v), x.scale, x.causal, x.window,
                             x.n_sink, rows=rows)
    if rows is not None:
        idx = torch.as_tensor(rows, dtype=torch.long, device=o.device)
        o = o.index_select(1, idx)
        lse = lse.index_select(2, idx)
    err = compare(o, lse, ro, rl, what, stress=stress)
    masked = np.isneginf(rl).transpose(0, 2, 1)  # [B, R, Hq]
    if masked.any():
        assert_masked_rows_zero(o, masked, what)
    return err


SMALL = [
    # (seed, B, Hq, Hkv, Sq, Skv, d, causal, window, n_sink, q_mult)
    (11, 1, 1, 1, 128, 128, 64, False, 0, 0, 1.0),      # the tiny configuration
    (12, 2, 3, 3, 300, 389, 128, False, 0, 0, 1.0),     # ragged, several tiles
    (13, 2, 2, 2, 640, 640, 128, True, 0, 0, 1.0),      # last CTA's second Q tile empty
    (14, 1, 2, 2, 333, 333, 128, True, 0, 0, 1.0),      # ragged causal
    (15, 1, 2, 2, 200, 700, 128, True, 0, 0, 1.0),      # Sq < Skv, shifted diagonal
    (16, 1, 2, 2, 500, 300, 128, True, 0, 0, 1.0),      # Sq > Skv: fully masked rows
    (17, 1, 2, 2, 512, 512, 128, False, 0, 0, 8.0),     # stress x8
    (18, 1, 2, 2, 512, 512, 128, True, 0, 0, 8.0),      # stress x8 causal
    (19, 1, 2, 2, 1500, 1500, 128, True, 300, 1, 1.0),  # window + one sink key
    (20, 1, 2, 2, 1100, 1100, 128, True, 128, 3, 1.0),  # narrow window, 3 sinks
    (21, 1, 2, 2, 700, 1000, 128, True, 64, 200, 1.0),  # sinks spanning tiles, Sq < Skv
    (22, 2, 8, 2, 700, 700, 128, True, 0, 0, 1.0),      # GQA 4:1
    (23, 1, 4, 1, 300, 300, 64, True, 0, 0, 1.0),       # d=64, MQA
    (24, 2, 2, 2, 257, 129, 64, False, 0, 0, 1.0),      # d=64 ragged non-causal
    (25, 1, 2, 2, 1, 1, 128, True, 0, 0, 1.0),          # single query, single key
    (26, 1, 2, 2, 129, 1, 128, True, 0, 0, 1.0),        # one key, most rows masked
]


@pytest.mark.parametrize("case", SMALL, ids=[f"seed{c[0]}" for c in SMALL])
def test_small_shapes(ea, case):
    seed, B, Hq, Hkv, Sq, Skv, d, causal, window, n_sink, qm = case
    x = workloads.dense_inputs(seed, B, Hq, Hkv, Sq, Skv, d, causal, window, n_sink, q_mult=qm)
    check_dense(ea, x, what=f"case seed {seed}", stress=qm != 1.0)


def test_empty_inputs(ea):
    # Sq == 0: nothing to do
    x = workloads.dense_inputs(31, 1, 2, 2, 0, 64, 128)
    o, lse = run_dense(ea, x)
    assert o.numel() == 0
    # Skv == 0: every row sees nothing
    x = workloads.dense_inputs(32, 2, 2, 2, 70, 0, 128)
    o, lse = run_dense(ea, x)
    assert torch.all(o.view(torch.int16) == 0)
    assert torch.all(torch.isneginf(lse))


def test_deterministic(ea):
    x = workloads.dense_inputs(33, 1, 4, 2, 900, 900, 128, True)
    o1, l1 = run_dense(ea, x)
    o2, l2 = run_dense(ea, x)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


@pytest.mark.parametrize("lq,lk,causal,window,n_sink", [
    ([1, 130, 257, 600, 77], None, True, 0, 0),
    ([300, 5, 129], [400, 5, 700], True, 0, 0),      # kv longer than q (cached prefix)
    ([300, 5, 129], [100, 50, 129], True, 0, 0),     # q longer than kv: masked rows
    ([200, 513, 64], [200, 300, 1], False, 0, 0),
    ([900, 333], None, True, 100, 2),
])
def test_varlen(ea, lq, lk, causal, window, n_sink):
    x = workloads.varlen_inputs(41, len(lq), 0, 0, 8, 2, 128, causal, window, n_sink,
                                lengths=lq, klengths=lk)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    o, lse = ea.attn_fwd_ex(q, k, v, x.cu_q.cuda(), x.cu_k.cuda(), max_seqlen_q=x.max_q,
                            max_seqlen_k=x.max_k, causal=causal, window=window, n_sink=n_sink,
                            scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    ro, rl = oracle.attn_fwd_varlen(np64(x.q), np64(x.k), np64(x.v), x.cu_q.numpy(),
                                    x.cu_k.numpy(), x.scale, causal, window, n_sink)
    compare(o, lse, ro, rl, "varlen")
    masked = np.isneginf(rl).T  # [Tq, Hq]
    if masked.any():
        assert_masked_rows_zero(o, masked, "varlen")


# ------------------------------------------------------------------ full sizes, sampled rows

@pytest.mark.parametrize("causal,stress", [(False, False), (True, False), (False, True),
                                           (True, True)])
def test_prefill_full_size(ea, causal, stress):
    x = workloads.prefill_mha(causal, stress)
    err = check_dense(ea, x, rows=sample_rows(2048), what=f"prefill c={causal} s={stress}",
                      stress=stress)
    print(f"prefill causal={causal} stress={stress}: max |dO| {err[0]:.2e}, max |dLSE| "
          f"{err[1]:.2e}, {err[2]} elements with |O| >= 4")


@pytest.mark.parametrize("window", [False, True])
def test_long_causal_full_size(ea, window):
    x = workloads.long_causal(window)
    rows = sample_rows(8192)
    if window:
        rows = np.unique(np.concatenate([rows, [1023, 1024, 1025, 2047, 2048]])).astype(np.int32)
    err = check_dense(ea, x, rows=rows, what=f"long window={window}")
    print(f"long causal window={window}: max |dO| {err[0]:.2e}, max |dLSE| {err[1]:.2e}, "
          f"{err[2]} elements with |O| >= 4")


def test_many_short_sequences(ea):
    """64 batch entries of 100 rows, GQA 4:1, causal: one partial Q tile per
    (batch, head), 512 items through the persistent grid."""
    x = workloads.dense_inputs(59, 64, 8, 2, 100, 100, 128, True)
    check_dense(ea, x, what="64 x 100 causal")


def test_very_long_causal(ea):
    """S = 32768 causal on two heads: items of up to 256 key tiles (the K/V
    ring, the tile counts and the item order far past the workloads'
    lengths), rows sampled in every tile."""
    x = workloads.dense_inputs(58, 1, 2, 2, 32768, 32768, 128, True)
    err = check_dense(ea, x, rows=sample_rows(32768), what="S=32768 causal")
    print(f"S=32768 causal: max |dO| {err[0]:.2e}, max |dLSE| {err[1]:.2e}")


def test_gqa_full_size(ea):
    x = workloads.gqa_causal()
    err = check_dense(ea, x, rows=sample_rows(4096), what="gqa")
    print(f"gqa causal: max |dO| {err[0]:.2e}, max |dLSE| {err[1]:.2e}, {err[2]} elements "
          f"with |O| >= 4")


def test_gqa_varlen_full_size(ea):
    x = workloads.gqa_varlen()
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    o, lse = ea.attn_fwd_ex(q, k, v, x.cu_q.cuda(), x.cu_k.cuda(), max_seqlen_q=x.max_q,
                            max_seqlen_k=x.max_k, causal=True, scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    cu = x.cu_q.tolist()
    worst = [0.0, 0.0, 0]
    for s in range(len(cu) - 1):
        a, e = cu[s], cu[s + 1]
        L = e - a
        rows = sample_rows(L, seed=s)
        ro, rl = oracle.attn_fwd(np64(x.q[None, a:e]), np64(x.k[None, a:e]), np64(x.v[None, a:e]),
                                 x.scale, True, rows=rows)
        idx = torch.as_tensor(rows.astype(np.int64) + a, device=o.device)
        err = compare(o.index_select(0, idx)[None], lse.index_select(1, idx)[None], ro, rl,
                      f"varlen seq {s}")
        worst = [max(worst[0], err[0]), max(worst[1], err[1]), worst[2] + err[2]]
    print(f"gqa varlen: max |dO| {worst[0]:.2e}, max |dLSE| {worst[1]:.2e}, {worst[2]} "
          f"elements with |O| >= 4")


def test_varlen_repeated_calls_report_ok(ea):
    """Packed GQA prefill mixes bulk and direct O stores within one CTA; a
    hand-off race between them once ended about one call in four in a bounded
    wait.  Thirty calls in a row must all report ATTN_OK."""
    x = workloads.gqa_varlen()
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    cu_q, cu_k = x.cu_q.cuda(), x.cu_k.cuda()
    o, lse = ea.attn_fwd_ex(q, k, v, cu_q, cu_k, max_seqlen_q=x.max_q, max_seqlen_k=x.max_k,
                            causal=True, scale=x.scale)
    for rep in range(30):
        ea.attn_fwd_ex(q, k, v, cu_q, cu_k, max_seqlen_q=x.max_q, max_seqlen_k=x.max_k, o=o,
                       lse=lse, causal=True, scale=x.scale)
        assert ea.attn_device_status() == ea.ATTN_OK, f"call {rep}"


@pytest.mark.parametrize("nseq,lo,hi,seed", [
    (40, 0, 700, 43),     # many short sequences, some empty: the dense item order
    (300, 1, 60, 44),     # more sequences than the dense order holds: the sparse order
])
def test_varlen_many_sequences(ea, nseq, lo, hi, seed):
    """Causal packed calls with many sequences of mixed lengths (zero-length
    ones included) against the oracle, every row."""
    x = workloads.varlen_inputs(seed, nseq, lo, hi, 4, 2, 128, causal=True)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    o, lse = ea.attn_fwd_ex(q, k, v, x.cu_q.cuda(), x.cu_k.cuda(), max_seqlen_q=x.max_q,
                            max_seqlen_k=x.max_k, causal=True, scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    ro, rl = oracle.attn_fwd_varlen(np64(x.q), np64(x.k), np64(x.v), x.cu_q.numpy(),
                                    x.cu_k.numpy(), x.scale, True)
    compare(o, lse, ro, rl, f"varlen {nseq} sequences")


def test_varlen_long_sequence(ea):
    """A packed causal call whose longest sequence has more than 64 query
    pairs (the sparse item order), beside short ones: sampled rows of the
    long sequence, every row of the others."""
    lq = [17000, 300, 1]
    x = workloads.varlen_inputs(46, len(lq), 0, 0, 2, 1, 128, causal=True, lengths=lq)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    o, lse = ea.attn_fwd_ex(q, k, v, x.cu_q.cuda(), x.cu_k.cuda(), max_seqlen_q=x.max_q,
                            max_seqlen_k=x.max_k, causal=True, scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    cu = x.cu_q.tolist()
    for s_, rows in ((0, sample_rows(lq[0], seed=46)), (1, None), (2, None)):
        a, e = cu[s_], cu[s_ + 1]
        ro, rl = oracle.attn_fwd(np64(x.q[None, a:e]), np64(x.k[None, a:e]),
                                 np64(x.v[None, a:e]), x.scale, True, rows=rows)
        idx = torch.as_tensor(a + (np.arange(e - a) if rows is None else np.asarray(rows)),
                              device=o.device)
        compare(o[None, idx], lse[None, :, idx], ro, rl, f"varlen long, sequence {s_}")


def test_varlen_sequences_without_keys(ea):
    """Causal packed sequences with no keys at all between ones with keys
    (items with query rows and no key tile, in the dense item order): O = 0
    and LSE = -inf there, the others as the oracle."""
    lq, lk = [200, 300, 150, 90], [0, 300, 0, 120]
    x = workloads.varlen_inputs(47, len(lq), 0, 0, 4, 2, 128, causal=True, lengths=lq,
                                klengths=lk)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    o, lse = ea.attn_fwd_ex(q, k, v, x.cu_q.cuda(), x.cu_k.cuda(), max_seqlen_q=x.max_q,
                            max_seqlen_k=x.max_k, causal=True, scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    ro, rl = oracle.attn_fwd_varlen(np64(x.q), np64(x.k), np64(x.v), x.cu_q.numpy(),
                                    x.cu_k.numpy(), x.scale, True)
    compare(o, lse, ro, rl, "varlen, sequences without keys")
    masked = np.isneginf(rl).T
    assert masked[:200].all() and masked[500:650].all()
    assert_masked_rows_zero(o, masked, "varlen, sequences without keys")


def test_varlen_bad_offsets_reported(ea):
    """A sequence whose offsets run backwards is reported as ATTN_ERR_BAD_INPUT
    and left out; a sequence before it is computed as usual."""
    x = workloads.varlen_inputs(45, 4, 0, 0, 4, 2, 128, causal=True, lengths=[100, 100, 100, 200])
    cu = x.cu_q.clone()
    cu[2] = 350   # sequence 1: 250 rows (> max_seqlen 200), sequence 2 runs backwards
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    o, lse = ea.attn_fwd_ex(q, k, v, cu.cuda(), cu.cuda(), max_seqlen_q=200, max_seqlen_k=200,
                            causal=True, scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_ERR_BAD_INPUT
    assert ea.attn_device_status() == ea.ATTN_OK  # cleared by the read
    ro, rl = oracle.attn_fwd(np64(x.q[None, :100]), np64(x.k[None, :100]), np64(x.v[None, :100]),
                             x.scale, True)
    compare(o[None, :100], lse[None, :, :100], ro, rl, "sequence 0 next to a bad one")
