"""Seeded random shapes through the forward, the decode and the backward
against the oracle: persistent grids with mixed item sizes, item records,
packed sequences, windows, sink keys and logit sinks in combinations the
fixed cases do not reach.  Each case draws its sizes from its own seed."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._parity import compare, np64, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ea():
    import exact_attention_08_gb300 as m
    assert torch.cuda.is_available()
    return m


def _draw(seed):
    r = np.random.default_rng(seed)
    Hkv = int(r.choice([1, 2, 4]))
    Hq = Hkv * int(r.choice([1, 2, 4]))
    causal = bool(r.random() < 0.7)
    window = int(r.choice([0, 0, 64, 300, 1000])) if causal else 0
    n_sink = int(r.choice([0, 1, 5])) if window else 0
    d = int(r.choice([64, 128, 128, 256]))
    return r, Hq, Hkv, causal, window, n_sink, d


@pytest.mark.parametrize("seed", range(301, 313))
def test_forward_dense(ea, seed):
    r, Hq, Hkv, causal, window, n_sink, d = _draw(seed)
    B = int(r.integers(1, 5))
    Sq = int(r.integers(1, 3000))
    Skv = Sq if r.random() < 0.5 else int(r.integers(1, 3000))
    x = workloads.dense_inputs(seed, B, Hq, Hkv, Sq, Skv, d, causal, window, n_sink)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    o, lse = ea.attn_fwd_ex(q, k, v, causal=causal, window=window, n_sink=n_sink, scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    rows = sample_rows(Sq, seed=seed)
    ro, rl = oracle.attn_fwd(np64(x.q), np64(x.k), np64(x.v), x.scale, causal, window, n_sink,
                             rows=rows)
    idx = torch.as_tensor(rows, dtype=torch.long, device=o.device)
    compare(o.index_select(1, idx), lse.index_select(2, idx), ro, rl,
            f"fuzz dense seed {seed} (B={B} Hq={Hq} Hkv={Hkv} Sq={Sq} Skv={Skv} d={d} "
            f"c={causal} w={window} s={n_sink})")


@pytest.mark.parametrize("seed", range(321, 331))
def test_forward_packed(ea, seed):
    r, Hq, Hkv, causal, window, n_sink, d = _draw(seed)
    nseq = int(r.integers(1, 40))
    lq = r.integers(0, 1500, nseq).tolist()
    lk = lq if r.random() < 0.6 else r.integers(0, 1500, nseq).tolist()
    x = workloads.varlen_inputs(seed, nseq, 0, 0, Hq, Hkv, d, causal, window, n_sink,
                                lengths=lq, klengths=lk)
    sink = workloads.logit_sinks(seed + 1, Hq) if r.random() < 0.3 else None
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    kw = dict(max_seqlen_q=x.max_q, max_seqlen_k=x.max_k, causal=causal, window=window,
              n_sink=n_sink, scale=x.scale)
    if sink is None:
        o, lse = ea.attn_fwd_ex(q, k, v, x.cu_q.cuda(), x.cu_k.cuda(), **kw)
    else:
        o, lse = ea.attn_fwd_ex_sink(q, k, v, sink.cuda(), x.cu_q.cuda(), x.cu_k.cuda(), **kw)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    ro, rl = oracle.attn_fwd_varlen(np64(x.q), np64(x.k), np64(x.v), x.cu_q.numpy(),
                                    x.cu_k.numpy(), x.scale, causal, window, n_sink,
                                    sink=None if sink is None else sink.double().numpy())
    compare(o, lse, ro, rl, f"fuzz packed seed {seed} (n={nseq} Hq={Hq} Hkv={Hkv} d={d} "
                            f"c={causal} w={window} s={n_sink} sink={sink is not None})")


@pytest.mark.parametrize("seed", range(341, 347))
def test_decode(ea, seed):
    r = np.random.default_rng(seed)
    Hkv = int(r.choice([1, 2, 8]))
    Hq = Hkv * int(r.choice([1, 4, 8]))
    d = int(r.choice([64, 128, 256]))
    B = int(r.integers(1, 80))
    splits = int(r.choice([1, 3, 8, 16]))
    x = workloads.paged_decode_inputs(seed, B, Hq, Hkv, d, 0, 3000, num_splits=splits)
    q, kp, vp = x.q.cuda(), x.k_pages.cuda(), x.v_pages.cuda()
    o, lse = ea.attn_decode_paged(q, kp, vp, x.page_table.cuda(), x.seqlens.cuda(),
                                  num_splits=splits, scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    req = list(range(B))
    k, v = x.contiguous_kv(req)
    ro, rl = oracle.attn_decode(np64(x.q), np64(k), np64(v), x.seqlens.numpy(), x.scale)
    compare(o, lse, ro, rl, f"fuzz decode seed {seed} (B={B} Hq={Hq} Hkv={Hkv} d={d} "
                            f"splits={splits})")


@pytest.mark.parametrize("seed", range(361, 365))
def test_backward(ea, seed):
    r = np.random.default_rng(seed)
    Hkv = int(r.choice([1, 2, 4]))
    Hq = Hkv * int(r.choice([1, 2]))
    causal = bool(r.random() < 0.6)
    window = int(r.choice([0, 200])) if causal else 0
    n_sink = int(r.choice([0, 3])) if window else 0
    d = int(r.choice([64, 128]))
    B = int(r.integers(1, 4))
    Sq = int(r.integers(1, 1200))
    Skv = Sq if r.random() < 0.5 else int(r.integers(1, 1200))
    x = workloads.dense_inputs(seed, B, Hq, Hkv, Sq, Skv, d, causal, window, n_sink)
    g = workloads.grad_output(seed + 50, x.q.shape)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    o, lse = ea.attn_fwd_ex(q, k, v, causal=causal, window=window, n_sink=n_sink, scale=x.scale)
    dq, dk, dv = ea.attn_bwd_ex(q, k, v, o, lse, g.cuda(), causal=causal, window=window,
                                n_sink=n_sink, scale=x.scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    rq, rk, rv = oracle.attn_bwd(np64(x.q), np64(x.k), np64(x.v), np64(g), x.scale, causal,
                                 window, n_sink)
    for a, b_, n in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
        ga = a.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(ga)), n
        scale = np.abs(b_).max()
        if scale == 0.0:
            assert np.abs(ga).max() <= 1e-4, n
            continue
        l2 = np.linalg.norm(ga - b_) / max(np.linalg.norm(b_), 1e-300)
        assert l2 <= 1e-2, f"fuzz backward seed {seed} {n}: relative L2 {l2:.3e}"
        assert np.abs(ga - b_).max() / scale <= 3e-2, f"fuzz backward seed {seed} {n}"


def _check_grads(seed, pairs, what):
    for a, b_, n in pairs:
        ga = a.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(ga)), n
        scale = np.abs(b_).max()
        if scale == 0.0:
            assert np.abs(ga).max() <= 1e-4, n
            continue
        l2 = np.linalg.norm(ga - b_) / max(np.linalg.norm(b_), 1e-300)
        assert l2 <= 1e-2, f"{what} seed {seed} {n}: relative L2 {l2:.3e}"


@pytest.mark.parametrize("seed", range(371, 377))
def test_backward_d256(ea, seed):
    """Head dimension 256 (three launches streaming 64-row tiles): dense or
    packed, with random lengths, masks and head groups."""
    r = np.random.default_rng(seed)
    Hkv = int(r.choice([1, 2]))
    Hq = Hkv * int(r.choice([1, 2, 4]))
    causal = bool(r.random() < 0.6)
    window = int(r.choice([0, 130])) if causal else 0
    n_sink = int(r.choice([0, 1, 65])) if window else 0
    if r.random() < 0.5:
        B = int(r.integers(1, 3))
        Sq = int(r.integers(1, 700))
        Skv = Sq if r.random() < 0.5 else int(r.integers(1, 700))
        x = workloads.dense_inputs(seed, B, Hq, Hkv, Sq, Skv, 256, causal, window, n_sink)
        g = workloads.grad_output(seed + 50, x.q.shape)
        q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
        o, lse = ea.attn_fwd_ex(q, k, v, causal=causal, window=window, n_sink=n_sink,
                                scale=x.scale)
        dq, dk, dv = ea.attn_bwd_ex(q, k, v, o, lse, g.cuda(), causal=causal, window=window,
                                    n_sink=n_sink, scale=x.scale)
        torch.cuda.synchronize()
        assert ea.attn_device_status() == ea.ATTN_OK
        ref = oracle.attn_bwd(np64(x.q), np64(x.k), np64(x.v), np64(g), x.scale, causal, window,
                              n_sink)
        _check_grads(seed, zip((dq, dk, dv), ref, ("dq", "dk", "dv")),
                     f"fuzz d=256 dense (B={B} Hq={Hq} Hkv={Hkv} Sq={Sq} Skv={Skv})")
        return
    nseq = int(r.integers(1, 5))
    lq = [int(v) for v in r.integers(1, 500, nseq)]
    lk = [int(v) for v in r.integers(1, 500, nseq)] if r.random() < 0.5 else None
    x = workloads.varlen_inputs(seed, nseq, 0, 0, Hq, Hkv, 256, causal, window, n_sink,
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
    for s in range(nseq):
        a, e, ka, ke = cu_q[s], cu_q[s + 1], cu_k[s], cu_k[s + 1]
        sq, sk, sv = oracle.attn_bwd(np64(x.q[None, a:e]), np64(x.k[None, ka:ke]),
                                     np64(x.v[None, ka:ke]), np64(g[None, a:e]), x.scale,
                                     causal, window, n_sink)
        rq[a:e], rk[ka:ke], rv[ka:ke] = sq[0], sk[0], sv[0]
    _check_grads(seed, ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")),
                 f"fuzz d=256 packed (lengths {lq} / {lk})")
