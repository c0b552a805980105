"""GPU parity of attn_bwd (through the C ABI) against the fp64 backward
oracle on the same seeded inputs.

Tolerance, from the arithmetic: P and dS enter the second products as bf16
(relative rounding 2^-9 each) and the gradients are returned in bf16 (2^-9);
accumulation is fp32.  Errors of that size average out over the 128+ terms
of each sum, so per tensor the relative L2 error must stay below 1e-2 (the
pages' own figure for a bf16, atomically accumulated dQ is 1.024 %, "TileLang
tutorial, ch.15", section 5.4) and the largest error below 3e-2 of the
tensor's largest magnitude."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._parity import np64

pytestmark = pytest.mark.gpu

REL_L2 = 1e-2
REL_MAX = 3e-2


@pytest.fixture(scope="module")
def ea():
    import exact_attention_08_gb300 as m
    assert torch.cuda.is_available()
    return m


def _run(ea, x, g):
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    o, lse = ea.attn_fwd_ex(q, k, v, causal=x.causal, scale=x.scale)
    dq, dk, dv = ea.attn_bwd(q, k, v, o, lse, g.cuda(), causal=x.causal, scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    return dq, dk, dv


def _check(got, ref, what):
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(g)), f"{what}: non-finite"
    scale = np.abs(ref).max()
    if scale == 0.0:
        # e.g. a single visible key: dS = P (dP - D) vanishes exactly, and the
        # kernel's D (from the bf16 O) and dP differ only by rounding
        assert np.abs(g).max() <= 1e-4, f"{what}: expected ~0, got {np.abs(g).max():.3e}"
        return 0.0, 0.0
    l2 = np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-300)
    mx = np.abs(g - ref).max() / scale
    assert l2 <= REL_L2, f"{what}: relative L2 error {l2:.3e}"
    assert mx <= REL_MAX, f"{what}: max error {mx:.3e} of the largest magnitude"
    return l2, mx


def _compare(ea, x, seed, what):
    g = workloads.grad_output(seed, x.q.shape)
    dq, dk, dv = _run(ea, x, g)
    rq, rk, rv = oracle.attn_bwd(np64(x.q), np64(x.k), np64(x.v), np64(g), x.scale, x.causal)
    return [_check(a, b, f"{what} {n}") for a, b, n in ((dq, rq, "dq"), (dk, rk, "dk"),
                                                          (dv, rv, "dv"))]


CASES = [
    # (seed, B, Hq, Hkv, Sq, Skv, d, causal)
    (101, 1, 1, 1, 128, 128, 64, False),
    (102, 2, 3, 3, 300, 389, 128, False),     # ragged, several tiles
    (103, 1, 2, 2, 333, 333, 128, True),      # ragged causal
    (104, 1, 2, 2, 200, 700, 128, True),      # Sq < Skv: shifted diagonal
    (105, 1, 2, 2, 500, 300, 128, True),      # Sq > Skv: rows with no key
    (106, 2, 8, 2, 400, 400, 128, True),      # GQA 4:1
    (107, 1, 4, 1, 300, 300, 64, True),       # d=64, MQA
    (108, 1, 2, 2, 1, 1, 128, True),          # one query, one key
]


@pytest.mark.parametrize("case", CASES, ids=[f"seed{c[0]}" for c in CASES])
def test_small(ea, case):
    seed, B, Hq, Hkv, Sq, Skv, d, causal = case
    x = workloads.dense_inputs(seed, B, Hq, Hkv, Sq, Skv, d, causal)
    _compare(ea, x, seed + 50, f"seed {seed}")


def test_rows_without_keys_get_zero_dq(ea):
    x = workloads.dense_inputs(109, 1, 2, 2, 300, 100, 128, True)
    g = workloads.grad_output(159, x.q.shape)
    dq, _, _ = _run(ea, x, g)
    assert torch.all(dq[:, :200].view(torch.int16) == 0)


def test_deterministic(ea):
    x = workloads.dense_inputs(110, 1, 4, 2, 700, 700, 128, True)
    g = workloads.grad_output(160, x.q.shape)
    a = _run(ea, x, g)
    b = _run(ea, x, g)
    for t1, t2 in zip(a, b):
        assert torch.equal(t1.view(torch.int16), t2.view(torch.int16))


def test_empty_sizes(ea):
    x = workloads.dense_inputs(111, 1, 2, 2, 0, 64, 128)  # no query: dk = dv = 0
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    o = torch.empty_like(q)
    lse = torch.empty(1, 2, 0, device="cuda")
    dk = torch.full_like(k, 3.0)
    dv = torch.full_like(v, 3.0)
    ea.attn_bwd(q, k, v, o, lse, torch.empty_like(q), dk=dk, dv=dv, scale=x.scale)
    torch.cuda.synchronize()
    assert torch.all(dk == 0) and torch.all(dv == 0)
    x = workloads.dense_inputs(112, 1, 2, 2, 70, 0, 128)  # no key: dq = 0
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    o, lse = ea.attn_fwd_ex(q, k, v, scale=x.scale)
    dq, _, _ = ea.attn_bwd(q, k, v, o, lse, workloads.grad_output(162, q.shape).cuda(),
                           scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    assert torch.all(dq.view(torch.int16) == 0)


@pytest.mark.parametrize("causal", [False, True])
def test_full_length(ea, causal):
    """S = 2048, d = 128 (the prefill workload's sequence length) on 4 heads."""
    x = workloads.dense_inputs(113 + int(causal), 1, 4, 4, 2048, 2048, 128, causal)
    errs = _compare(ea, x, 163 + int(causal), f"S=2048 causal={causal}")
    print("bwd rel L2 / max:", errs)


def test_long_causal(ea):
    """S = 8192 causal on two heads (the long-sequence shape): 64 key tiles a
    head, so every CTA of the persistent grids walks one long item through
    the operand rings (every element compared)."""
    x = workloads.dense_inputs(115, 1, 2, 2, 8192, 8192, 128, True)
    errs = _compare(ea, x, 165, "S=8192 causal")
    print("bwd S=8192 rel L2 / max:", errs)


# ------------------------------------------------------------------ sink keys, window, packed

WINDOW_CASES = [
    # (seed, B, Hq, Hkv, Sq, Skv, d, window, n_sink)
    (121, 1, 2, 2, 700, 700, 128, 200, 1),      # window + one sink key
    (122, 1, 4, 2, 600, 900, 128, 100, 3),      # Sq < Skv, GQA
    (123, 1, 2, 2, 1500, 1500, 64, 300, 130),   # sinks spanning two key tiles, d=64
    (124, 1, 2, 2, 500, 300, 128, 64, 2),       # Sq > Skv: rows with no key
    (125, 2, 2, 2, 400, 400, 128, 128, 0),      # window alone, tile-aligned
]


@pytest.mark.parametrize("case", WINDOW_CASES, ids=[f"seed{c[0]}" for c in WINDOW_CASES])
def test_window_and_sink_keys(ea, case):
    """Causal sliding window with sink keys (attn_bwd_ex) against the oracle."""
    seed, B, Hq, Hkv, Sq, Skv, d, window, n_sink = case
    x = workloads.dense_inputs(seed, B, Hq, Hkv, Sq, Skv, d, True, window, n_sink)
    g = workloads.grad_output(seed + 50, x.q.shape)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    o, lse = ea.attn_fwd_ex(q, k, v, causal=True, window=window, n_sink=n_sink, scale=x.scale)
    dq, dk, dv = ea.attn_bwd_ex(q, k, v, o, lse, g.cuda(), causal=True, window=window,
                                n_sink=n_sink, scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    rq, rk, rv = oracle.attn_bwd(np64(x.q), np64(x.k), np64(x.v), np64(g), x.scale, True, window,
                                 n_sink)
    for a, b, n in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
        _check(a, b, f"window seed {seed} {n}")


VARLEN_CASES = [
    # (seed, query lengths, key lengths (None: the same), Hq, Hkv, causal, window, n_sink)
    (131, [300, 1, 129, 700, 256], None, 8, 2, True, 0, 0),
    (132, [200, 5, 129], [400, 5, 700], 4, 4, True, 0, 0),     # cached prefixes (Sq < Skv)
    (133, [150, 64, 300], [100, 64, 1], 4, 2, True, 0, 0),     # Sq > Skv: rows with no key
    (134, [200, 513, 64], [200, 300, 1], 4, 2, False, 0, 0),
    (135, [900, 333], None, 4, 2, True, 100, 2),               # window + sink keys
]


@pytest.mark.parametrize("case", VARLEN_CASES, ids=[f"seed{c[0]}" for c in VARLEN_CASES])
def test_varlen(ea, case):
    """Packed sequences (cu_seqlens) against the oracle, sequence by sequence."""
    seed, lq, lk, Hq, Hkv, causal, window, n_sink = case
    x = workloads.varlen_inputs(seed, len(lq), 0, 0, Hq, Hkv, 128, causal, window, n_sink,
                                lengths=lq, klengths=lk)
    g = workloads.grad_output(seed + 50, x.q.shape)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    cq, ck = x.cu_q.cuda(), x.cu_k.cuda()
    o, lse = ea.attn_fwd_ex(q, k, v, cq, ck, max_seqlen_q=x.max_q, max_seqlen_k=x.max_k,
                            causal=causal, window=window, n_sink=n_sink, scale=x.scale)
    dq, dk, dv = ea.attn_bwd_ex(q, k, v, o, lse, g.cuda(), cq, ck, max_seqlen_q=x.max_q,
                                max_seqlen_k=x.max_k, causal=causal, window=window,
                                n_sink=n_sink, scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    cu_q, cu_k = x.cu_q.tolist(), x.cu_k.tolist()
    rq = np.zeros(x.q.shape)
    rk = np.zeros(x.k.shape)
    rv = np.zeros(x.v.shape)
    for s in range(len(lq)):
        a, e, ka, ke = cu_q[s], cu_q[s + 1], cu_k[s], cu_k[s + 1]
        sq, sk, sv = oracle.attn_bwd(np64(x.q[None, a:e]), np64(x.k[None, ka:ke]),
                                     np64(x.v[None, ka:ke]), np64(g[None, a:e]), x.scale,
                                     causal, window, n_sink)
        rq[a:e], rk[ka:ke], rv[ka:ke] = sq[0], sk[0], sv[0]
    for a_, b_, n in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
        _check(a_, b_, f"varlen seed {seed} {n}")


def test_varlen_matches_dense(ea):
    """One packed sequence gives the same bits as the dense call."""
    x = workloads.dense_inputs(136, 1, 4, 2, 500, 500, 128, True)
    g = workloads.grad_output(186, x.q.shape).cuda()
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    o, lse = ea.attn_fwd(q, k, v, causal=True, scale=x.scale)
    dense = ea.attn_bwd(q, k, v, o, lse, g, causal=True, scale=x.scale)
    cu = torch.tensor([0, 500], dtype=torch.int32, device="cuda")
    packed = ea.attn_bwd_ex(q[0], k[0], v[0], o[0], lse[0].contiguous(), g[0], cu, cu,
                            max_seqlen_q=500, max_seqlen_k=500, causal=True, scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    for a, b in zip(dense, packed):
        assert torch.equal(a[0].view(torch.int16), b.view(torch.int16))


def _dsink_bound(o, lse, g, sink):
    """Per-head tolerance on the sink gradient, from the arithmetic: the
    kernel forms D = rowsum(dO * O) from the bf16 O, each element with an
    independent relative rounding of at most 2^-9, so the error of
    sum_rows P_sink D has a standard deviation of about
    2^-9 / sqrt(3) * sqrt(sum_rows P_sink^2 sum_t (dO_t O_t)^2); the bound
    takes 8 of those (about 14 sigma) plus 1e-3 of sum_rows P_sink |D| for the
    fp32 LSE that P_sink is rebuilt from (dense [B,Sq,Hq,d] / [B,Hq,Sq] fp64
    arrays from the oracle)."""
    p = np.exp(np.asarray(sink, np.float64)[None, :, None] - lse)        # [B, Hq, Sq]
    p = np.where(np.isfinite(p), p, 0.0)
    go = (g * o).transpose(0, 2, 1, 3)                                    # [B, Hq, Sq, d]
    rnd = np.sqrt(np.sum(p ** 2 * np.sum(go ** 2, axis=-1), axis=(0, 2)))
    lsee = np.sum(p * np.abs(go.sum(axis=-1)), axis=(0, 2))
    return 8.0 * 2.0 ** -9 * rnd + 1e-3 * lsee + 1e-6


def _check_dsink(got, ref, bound, what):
    got = got.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite"
    err = np.abs(got - ref)
    assert np.all(err <= bound), f"{what}: errors {err} above {bound}"


SINK_CASES = [
    # (seed, B, Hq, Hkv, Sq, Skv, d, causal, window, n_sink, extreme sinks)
    (141, 2, 4, 2, 300, 300, 128, True, 0, 0, True),    # -inf, +100, -30 and a plain sink
    (142, 1, 4, 4, 400, 700, 64, False, 0, 0, False),   # non-causal, d=64
    (143, 1, 4, 2, 600, 600, 128, True, 128, 2, False),  # window + sink keys
    (144, 1, 2, 2, 500, 300, 128, True, 0, 0, False),   # Sq > Skv: rows with no key
]


@pytest.mark.parametrize("case", SINK_CASES, ids=[f"seed{c[0]}" for c in SINK_CASES])
def test_logit_sink(ea, case):
    """attn_bwd_ex_sink: dq, dk, dv and the sink's gradient against the
    oracle's backward with the same logit sink."""
    seed, B, Hq, Hkv, Sq, Skv, d, causal, window, n_sink, extremes = case
    x = workloads.dense_inputs(seed, B, Hq, Hkv, Sq, Skv, d, causal, window, n_sink)
    g = workloads.grad_output(seed + 50, x.q.shape)
    sink = workloads.logit_sinks(seed + 70, Hq, extremes=extremes)
    q, k, v, sg = x.q.cuda(), x.k.cuda(), x.v.cuda(), sink.cuda()
    o, lse = ea.attn_fwd_ex_sink(q, k, v, sg, causal=causal, window=window, n_sink=n_sink,
                                 scale=x.scale)
    dq, dk, dv, ds = ea.attn_bwd_ex_sink(q, k, v, o, lse, g.cuda(), sg, causal=causal,
                                         window=window, n_sink=n_sink, scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    rq, rk, rv, rs = oracle.attn_bwd(np64(x.q), np64(x.k), np64(x.v), np64(g), x.scale, causal,
                                     window, n_sink, sink=sink.double().numpy())
    for a, b, n in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
        _check(a, b, f"sink seed {seed} {n}")
    ro, rl = oracle.attn_fwd(np64(x.q), np64(x.k), np64(x.v), x.scale, causal, window, n_sink,
                             sink=sink.double().numpy())
    _check_dsink(ds, rs, _dsink_bound(ro, rl, np64(g), sink.numpy()), f"sink seed {seed} dsink")
    if extremes:
        assert ds[0].item() == 0.0  # sigma = -inf: no sink, no gradient
    # a fixed summation order: the same bits again
    again = ea.attn_bwd_ex_sink(q, k, v, o, lse, g.cuda(), sg, causal=causal, window=window,
                                n_sink=n_sink, scale=x.scale)
    torch.cuda.synchronize()
    assert torch.equal(again[3], ds)
    assert torch.equal(again[0].view(torch.int16), dq.view(torch.int16))


def test_logit_sink_varlen(ea):
    """Packed sequences with a logit sink: the sink's gradient sums every
    sequence's rows of the head."""
    lq, lk = [300, 1, 129, 500], [300, 40, 129, 200]
    Hq, Hkv = 4, 2
    x = workloads.varlen_inputs(145, len(lq), 0, 0, Hq, Hkv, 128, True, lengths=lq, klengths=lk)
    g = workloads.grad_output(195, x.q.shape)
    sink = workloads.logit_sinks(215, Hq)
    q, k, v, sg = x.q.cuda(), x.k.cuda(), x.v.cuda(), sink.cuda()
    cq, ck = x.cu_q.cuda(), x.cu_k.cuda()
    o, lse = ea.attn_fwd_ex_sink(q, k, v, sg, cq, ck, max_seqlen_q=x.max_q, max_seqlen_k=x.max_k,
                                 causal=True, scale=x.scale)
    dq, dk, dv, ds = ea.attn_bwd_ex_sink(q, k, v, o, lse, g.cuda(), sg, cq, ck,
                                         max_seqlen_q=x.max_q, max_seqlen_k=x.max_k, causal=True,
                                         scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    cu_q, cu_k = x.cu_q.tolist(), x.cu_k.tolist()
    rq, rk, rv = np.zeros(x.q.shape), np.zeros(x.k.shape), np.zeros(x.v.shape)
    rs = np.zeros(Hq)
    os_, ls_, gs_ = [], [], []
    sk = sink.double().numpy()
    for s in range(len(lq)):
        a, e, ka, ke = cu_q[s], cu_q[s + 1], cu_k[s], cu_k[s + 1]
        qs, ks, vs, gs = (np64(x.q[None, a:e]), np64(x.k[None, ka:ke]), np64(x.v[None, ka:ke]),
                          np64(g[None, a:e]))
        sq, skk, sv, sds = oracle.attn_bwd(qs, ks, vs, gs, x.scale, True, sink=sk)
        rq[a:e], rk[ka:ke], rv[ka:ke] = sq[0], skk[0], sv[0]
        rs += sds
        ro, rl = oracle.attn_fwd(qs, ks, vs, x.scale, True, sink=sk)
        os_.append(ro[0])
        ls_.append(rl[0])
        gs_.append(gs[0])
    for a_, b_, n in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
        _check(a_, b_, f"varlen sink {n}")
    # the packed rows as one batch row: [1, Tq, Hq, d] and [1, Hq, Tq]
    bound = _dsink_bound(np.concatenate(os_)[None], np.concatenate(ls_, axis=1)[None],
                         np.concatenate(gs_)[None], sk)
    _check_dsink(ds, rs, bound, "varlen sink dsink")


def test_logit_sink_without_queries(ea):
    """No query row: dk = dv = 0 and a zero sink gradient."""
    q = torch.zeros(1, 0, 2, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.randn(1, 5, 2, 128, device="cuda").to(torch.bfloat16)
    lse = torch.zeros(1, 2, 0, device="cuda")
    sg = torch.tensor([1.0, 2.0], device="cuda")
    ds = torch.full((2,), 7.0, device="cuda")
    dq, dk, dv, ds = ea.attn_bwd_ex_sink(q, k, k, q, lse, q, sg, dsink=ds, causal=True)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dk) == 0 and torch.count_nonzero(dv) == 0
    assert torch.count_nonzero(ds) == 0


PERSISTENT_CASES = [
    # (seed, B, Hq, Hkv, Sq, Skv, causal, window, n_sink): more key tiles and
    # query tiles than SMs, so every CTA of the persistent grids walks
    # several items, some of which have no tile to process
    (151, 4, 8, 8, 1500, 1024, True, 0, 0),     # Sq > Skv: query tiles with no key
    (152, 4, 8, 4, 300, 2048, True, 100, 2),    # key tiles no query sees (window)
]


@pytest.mark.parametrize("case", PERSISTENT_CASES, ids=[f"seed{c[0]}" for c in PERSISTENT_CASES])
def test_persistent_items(ea, case):
    """Dense calls large enough that the persistent dK/dV and dQ grids give
    each CTA several items, empty ones among them, against the oracle."""
    seed, B, Hq, Hkv, Sq, Skv, causal, window, n_sink = case
    x = workloads.dense_inputs(seed, B, Hq, Hkv, Sq, Skv, 128, causal, window, n_sink)
    g = workloads.grad_output(seed + 50, x.q.shape)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    o, lse = ea.attn_fwd_ex(q, k, v, causal=causal, window=window, n_sink=n_sink, scale=x.scale)
    dq, dk, dv = ea.attn_bwd_ex(q, k, v, o, lse, g.cuda(), causal=causal, window=window,
                                n_sink=n_sink, scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    rq, rk, rv = oracle.attn_bwd(np64(x.q), np64(x.k), np64(x.v), np64(g), x.scale, causal, window,
                                 n_sink)
    for a, b, n in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
        _check(a, b, f"persistent seed {seed} {n}")
    # exact zeros where nothing is seen: query rows before the first key,
    # keys no query's window reaches
    if Sq > Skv:
        assert torch.count_nonzero(dq[:, :Sq - Skv]) == 0
    if window > 0:
        first_seen = Skv - Sq - window + 1  # the first window key of query 0
        assert torch.count_nonzero(dk[:, n_sink:first_seen]) == 0
        assert torch.count_nonzero(dv[:, n_sink:first_seen]) == 0


@pytest.mark.parametrize("d", [128, 256])
def test_stream_order_after_launch_chain(ea, d):
    """Work queued on the stream after attn_bwd sees every gradient complete.
    The gradient kernels run as a programmatic launch chain (each may start
    while the one before it drains), so the last kernel's completion has to
    imply the earlier ones': copies taken on the same stream, with no host
    synchronisation in between, must equal the gradients."""
    x = workloads.dense_inputs(113, 4, 16, 16, 2048, 2048, d, False)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    g = workloads.grad_output(163, x.q.shape).cuda()
    o, lse = ea.attn_fwd_ex(q, k, v, scale=x.scale)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dq, dk, dv = ea.attn_bwd(q, k, v, o, lse, g, scale=x.scale, stream=s)
        copies = [t.clone() for t in (dv, dk, dq)]
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    for c, t in zip(copies, (dv, dk, dq)):
        assert torch.equal(c.view(torch.int16), t.view(torch.int16))
    assert torch.count_nonzero(dv) > 0
