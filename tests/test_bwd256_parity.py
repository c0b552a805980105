"""GPU parity of the backward at head dimension 256 (attn_bwd, attn_bwd_ex,
attn_bwd_ex_sink through the C ABI) against the fp64 backward oracle on the
same seeded inputs, with the tolerance of the d = 64 / 128 tests (derived
there).  At d = 256 the gradients come from three launches (dV, dK, dQ)
that stream 64-row tiles, so the cases put tile and sequence boundaries at
multiples of 64 and off them, and give some key tiles no query and some
query rows no key."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._parity import np64
from tests.test_bwd_parity import _check, _check_dsink, _dsink_bound

pytestmark = pytest.mark.gpu

D = 256


@pytest.fixture(scope="module")
def ea():
    import exact_attention_08_gb300 as m
    assert torch.cuda.is_available()
    return m


def _dense(ea, x, g, window=0, n_sink=0):
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    o, lse = ea.attn_fwd_ex(q, k, v, causal=x.causal, window=window, n_sink=n_sink,
                            scale=x.scale)
    dq, dk, dv = ea.attn_bwd_ex(q, k, v, o, lse, g.cuda(), causal=x.causal, window=window,
                                n_sink=n_sink, scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    return dq, dk, dv


CASES = [
    # (seed, B, Hq, Hkv, Sq, Skv, causal, window, n_sink)
    (201, 1, 1, 1, 128, 128, False, 0, 0),      # one tile each way
    (202, 2, 3, 3, 300, 389, False, 0, 0),      # ragged, several tiles
    (203, 1, 2, 2, 333, 333, True, 0, 0),       # ragged causal
    (204, 1, 2, 2, 200, 700, True, 0, 0),       # Sq < Skv: shifted diagonal
    (205, 1, 2, 2, 500, 300, True, 0, 0),       # Sq > Skv: rows with no key
    (206, 2, 8, 2, 400, 400, True, 0, 0),       # GQA 4:1
    (207, 1, 4, 1, 257, 257, True, 0, 0),       # MQA, one row past a 256 boundary
    (208, 1, 2, 2, 1, 1, True, 0, 0),           # one query, one key
    (209, 1, 2, 2, 700, 700, True, 200, 1),     # window + one sink key
    (210, 1, 4, 2, 600, 900, True, 100, 3),     # window, Sq < Skv, GQA
    (211, 1, 2, 2, 900, 900, True, 150, 70),    # sinks spanning two 64-key tiles
    (212, 1, 2, 2, 500, 300, True, 64, 2),      # window, Sq > Skv
    (213, 2, 2, 2, 384, 384, True, 128, 0),     # window alone, tile-aligned
]


@pytest.mark.parametrize("case", CASES, ids=[f"seed{c[0]}" for c in CASES])
def test_dense(ea, case):
    seed, B, Hq, Hkv, Sq, Skv, causal, window, n_sink = case
    x = workloads.dense_inputs(seed, B, Hq, Hkv, Sq, Skv, D, causal, window, n_sink)
    g = workloads.grad_output(seed + 50, x.q.shape)
    got = _dense(ea, x, g, window, n_sink)
    ref = oracle.attn_bwd(np64(x.q), np64(x.k), np64(x.v), np64(g), x.scale, causal, window,
                          n_sink)
    for a, b, n in zip(got, ref, ("dq", "dk", "dv")):
        _check(a, b, f"d=256 seed {seed} {n}")


@pytest.mark.parametrize("causal", [False, True])
def test_full_length(ea, causal):
    """S = 2048 on two heads: 32 query tiles and 16 key tiles per head."""
    x = workloads.dense_inputs(221 + int(causal), 1, 2, 2, 2048, 2048, D, causal)
    g = workloads.grad_output(271 + int(causal), x.q.shape)
    got = _dense(ea, x, g)
    ref = oracle.attn_bwd(np64(x.q), np64(x.k), np64(x.v), np64(g), x.scale, causal)
    errs = [_check(a, b, f"d=256 S=2048 causal={causal} {n}")
            for a, b, n in zip(got, ref, ("dq", "dk", "dv"))]
    print("d=256 bwd rel L2 / max:", errs)


def test_exact_zeros(ea):
    """Query rows before the first visible key get dq = 0, keys that no
    query sees (past the window) get dk = dv = 0 (a row whose tile has
    visible pairs sums exact zero products, which may carry a sign)."""
    x = workloads.dense_inputs(223, 1, 2, 2, 300, 100, D, True)  # rows 0..199 see no key
    g = workloads.grad_output(273, x.q.shape)
    dq, _, _ = _dense(ea, x, g)
    assert torch.count_nonzero(dq[:, :200]) == 0
    x = workloads.dense_inputs(224, 1, 2, 2, 100, 1000, D, True, 64, 0)  # keys < 836 unseen
    g = workloads.grad_output(274, x.q.shape)
    _, dk, dv = _dense(ea, x, g, 64, 0)
    assert torch.count_nonzero(dk[:, :836]) == 0
    assert torch.count_nonzero(dv[:, :836]) == 0


def test_deterministic(ea):
    x = workloads.dense_inputs(225, 1, 4, 2, 700, 700, D, True)
    g = workloads.grad_output(275, x.q.shape)
    a = _dense(ea, x, g)
    b = _dense(ea, x, g)
    for t1, t2 in zip(a, b):
        assert torch.equal(t1.view(torch.int16), t2.view(torch.int16))


VARLEN_CASES = [
    # (seed, query lengths, key lengths (None: the same), Hq, Hkv, causal, window, n_sink)
    (231, [300, 1, 129, 700, 256], None, 4, 2, True, 0, 0),
    (232, [200, 5, 129], [400, 5, 700], 4, 4, True, 0, 0),     # cached prefixes (Sq < Skv)
    (233, [150, 64, 300], [100, 64, 1], 4, 2, True, 0, 0),     # Sq > Skv: rows with no key
    (234, [200, 513, 64], [200, 300, 1], 2, 2, False, 0, 0),
    (235, [900, 333], None, 4, 2, True, 100, 2),               # window + sink keys
]


@pytest.mark.parametrize("case", VARLEN_CASES, ids=[f"seed{c[0]}" for c in VARLEN_CASES])
def test_varlen(ea, case):
    """Packed sequences: rows of the next sequence share the last tiles."""
    seed, lq, lk, Hq, Hkv, causal, window, n_sink = case
    x = workloads.varlen_inputs(seed, len(lq), 0, 0, Hq, Hkv, D, causal, window, n_sink,
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
    rq, rk, rv = np.zeros(x.q.shape), np.zeros(x.k.shape), np.zeros(x.v.shape)
    for s in range(len(lq)):
        a, e, ka, ke = cu_q[s], cu_q[s + 1], cu_k[s], cu_k[s + 1]
        sq, sk, sv = oracle.attn_bwd(np64(x.q[None, a:e]), np64(x.k[None, ka:ke]),
                                     np64(x.v[None, ka:ke]), np64(g[None, a:e]), x.scale,
                                     causal, window, n_sink)
        rq[a:e], rk[ka:ke], rv[ka:ke] = sq[0], sk[0], sv[0]
    for a_, b_, n in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
        _check(a_, b_, f"d=256 varlen seed {seed} {n}")


def test_logit_sink(ea):
    """attn_bwd_ex_sink at d = 256: the sink's gradient comes from the row
    statistics the d = 256 kernels share with the others."""
    seed, B, Hq, Hkv, Sq, Skv = 241, 2, 4, 2, 300, 300
    x = workloads.dense_inputs(seed, B, Hq, Hkv, Sq, Skv, D, True)
    g = workloads.grad_output(seed + 50, x.q.shape)
    sink = workloads.logit_sinks(seed + 70, Hq, extremes=True)
    q, k, v, sg = x.q.cuda(), x.k.cuda(), x.v.cuda(), sink.cuda()
    o, lse = ea.attn_fwd_ex_sink(q, k, v, sg, causal=True, scale=x.scale)
    dq, dk, dv, ds = ea.attn_bwd_ex_sink(q, k, v, o, lse, g.cuda(), sg, causal=True,
                                         scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    rq, rk, rv, rs = oracle.attn_bwd(np64(x.q), np64(x.k), np64(x.v), np64(g), x.scale, True,
                                     sink=sink.double().numpy())
    for a, b, n in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
        _check(a, b, f"d=256 sink {n}")
    ro, rl = oracle.attn_fwd(np64(x.q), np64(x.k), np64(x.v), x.scale, True,
                             sink=sink.double().numpy())
    _check_dsink(ds, rs, _dsink_bound(ro, rl, np64(g), sink.numpy()), "d=256 dsink")
    assert ds[0].item() == 0.0


def test_empty_sizes(ea):
    """No query: dk = dv = 0; no key: dq = 0."""
    x = workloads.dense_inputs(242, 1, 2, 2, 0, 64, D)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    dk = torch.full_like(k, 3.0)
    dv = torch.full_like(v, 3.0)
    ea.attn_bwd(q, k, v, torch.empty_like(q), torch.empty(1, 2, 0, device="cuda"),
                torch.empty_like(q), dk=dk, dv=dv, scale=x.scale)
    torch.cuda.synchronize()
    assert torch.all(dk == 0) and torch.all(dv == 0)
    x = workloads.dense_inputs(243, 1, 2, 2, 70, 0, D)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    o, lse = ea.attn_fwd_ex(q, k, v, scale=x.scale)
    dq, _, _ = ea.attn_bwd(q, k, v, o, lse, workloads.grad_output(293, q.shape).cuda(),
                           scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    assert torch.all(dq.view(torch.int16) == 0)
