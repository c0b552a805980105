"""Pins for the oracle's logit sink ("TileLang tutorial, ch.15 Operators:
Attention", section 4.6: the attention-sink variant adds one term to the
softmax denominator in the epilogue, taken against m* = max(sink, m)).

Reading: the sink of query head h is a logit sigma_h in the units of
S = scale * Q K^T (natural log) that joins each row's softmax as one more
column with a zero value row; sigma_h = -inf is no sink.  The oracle's two
formulations (an extra column in the two-pass definition, an epilogue term
after the blockwise recurrence) and an independent brute force are checked
against each other and against closed forms, so that a plausible slip (sink
left out of the maximum, added to the numerator, scaled by `scale` again,
taken in base 2, or given a value row) fails at least one pin.
"""
import math

import numpy as np
import pytest

import oracle
from tests import _bruteforce as bf


def _rand(rng, B, Sq, Skv, Hq, Hkv, d, qmul=1.0):
    return (rng.normal(size=(B, Sq, Hq, d)) * qmul, rng.normal(size=(B, Skv, Hkv, d)),
            rng.normal(size=(B, Skv, Hkv, d)))


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


MODES = [(False, 0, 0), (True, 0, 0), (True, 3, 1)]


@pytest.mark.parametrize("causal,window,n_sink", MODES)
def test_minus_inf_sink_is_no_sink(causal, window, n_sink):
    """sigma = -inf everywhere reproduces the sink-free results bit for bit."""
    rng = np.random.default_rng(101)
    q, k, v = _rand(rng, 2, 7, 9, 4, 2, 8)
    none = np.full(4, -np.inf)
    a = oracle.attn_fwd(q, k, v, 0.4, causal, window, n_sink)
    b = oracle.attn_fwd(q, k, v, 0.4, causal, window, n_sink, sink=none)
    c = oracle.attn_fwd_blockwise(q, k, v, 0.4, causal, window, n_sink, block=4, sink=none)
    d = oracle.attn_fwd_blockwise(q, k, v, 0.4, causal, window, n_sink, block=4)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    assert all(np.array_equal(x, y) for x, y in zip(c, d))


@pytest.mark.parametrize("mode", ["full", "causal", "window_sink"])
def test_zero_keys_closed_form(mode):
    """K = 0: every visible logit is 0, so with n visible keys
    O = (sum of their V rows) / (n + e^sigma) and LSE = ln(n + e^sigma)."""
    Sq, Skv, d, Hq = 7, 10, 4, 3
    causal = mode != "full"
    window, n_sink = (3, 2) if mode == "window_sink" else (0, 0)
    rng = np.random.default_rng(102)
    q = rng.normal(size=(1, Sq, Hq, d))
    k = np.zeros((1, Skv, Hq, d))
    v = rng.normal(size=(1, Skv, Hq, d))
    sg = np.array([-1.5, 0.0, 2.25])
    o, lse = oracle.attn_fwd(q, k, v, 0.5, causal, window, n_sink, sink=sg)
    off = Skv - Sq
    for h in range(Hq):
        for i in range(Sq):
            vis = [j for j in range(Skv)
                   if (not causal or j <= i + off)
                   and (window == 0 or j > i + off - window or j < n_sink)]
            z = len(vis) + math.exp(sg[h])
            np.testing.assert_allclose(o[0, i, h], v[0, vis, h].sum(0) / z, rtol=0, atol=1e-14)
            assert abs(lse[0, h, i] - math.log(z)) < 1e-14


def test_one_key_is_logistic_in_key_minus_sink():
    """One key of logit a and a sink sigma: O = V_0 * sigmoid(a - sigma) and
    LSE = ln(e^a + e^sigma)."""
    d = 3
    q = np.array([1.0, 0.0, 0.0]).reshape(1, 1, 1, d)
    k = np.array([0.8, 4.0, -2.0]).reshape(1, 1, 1, d)
    v = np.array([2.0, -1.0, 0.5]).reshape(1, 1, 1, d)
    s, sg = 1.5, 0.3
    a = s * 0.8
    o, lse = oracle.attn_fwd(q, k, v, s, sink=[sg])
    w = 1.0 / (1.0 + math.exp(sg - a))
    np.testing.assert_allclose(o[0, 0, 0], w * v[0, 0, 0], rtol=0, atol=1e-15)
    assert abs(lse[0, 0, 0] - math.log(math.exp(a) + math.exp(sg))) < 1e-15


@pytest.mark.parametrize("causal,window,n_sink", MODES + [(True, 0, 0)])
def test_identity_against_sink_free_oracle(causal, window, n_sink):
    """The sink only enlarges the denominator: with O, LSE the sink-free
    results, O_sink = O * sigmoid(LSE - sigma) and LSE_sink = logaddexp(LSE, sigma)."""
    rng = np.random.default_rng(103)
    q, k, v = _rand(rng, 2, 9, 12, 6, 3, 8, qmul=2.0)
    sg = np.array([-np.inf, -3.0, 0.0, 1.7, 6.0, 40.0])
    o, lse = oracle.attn_fwd(q, k, v, 0.45, causal, window, n_sink)
    os_, ls = oracle.attn_fwd(q, k, v, 0.45, causal, window, n_sink, sink=sg)
    fac = _sigmoid(lse - sg[None, :, None])          # [B, Hq, Sq]
    np.testing.assert_allclose(os_, o * fac.transpose(0, 2, 1)[..., None], rtol=0, atol=1e-13)
    np.testing.assert_allclose(ls, np.logaddexp(lse, sg[None, :, None]), rtol=0, atol=1e-13)


def test_no_visible_key_gives_zero_and_the_sink():
    """A row that sees no key (causal with Sq > Skv, or Skv = 0) but has a
    finite sink: O = +0.0 and LSE = sigma exactly; with sigma = -inf it stays
    O = 0, LSE = -inf."""
    rng = np.random.default_rng(104)
    Sq, Skv = 9, 3
    q, k, v = _rand(rng, 1, Sq, Skv, 2, 2, 8)
    sg = np.array([0.625, -np.inf])
    for fn in (lambda: oracle.attn_fwd(q, k, v, 0.4, True, sink=sg),
               lambda: oracle.attn_fwd_blockwise(q, k, v, 0.4, True, block=2, sink=sg)):
        o, lse = fn()
        assert np.all(o[0, : Sq - Skv] == 0.0) and not np.signbit(o[0, : Sq - Skv]).any()
        assert np.all(lse[0, 0, : Sq - Skv] == 0.625)
        assert np.all(np.isneginf(lse[0, 1, : Sq - Skv]))
    q0, k0, v0 = q, k[:, :0], v[:, :0]
    o, lse = oracle.attn_fwd(q0, k0, v0, 0.4, sink=sg)
    assert np.all(o == 0.0) and np.all(lse[0, 0] == 0.625) and np.all(np.isneginf(lse[0, 1]))


def test_dominant_sink_stays_finite():
    """A sink far above every logit (e^sigma overflows fp64): O is ~0, LSE is
    sigma, and nothing is inf or nan (the m* = max(sink, m) reference)."""
    rng = np.random.default_rng(105)
    q, k, v = _rand(rng, 1, 5, 7, 2, 1, 4)
    sg = np.array([800.0, 750.0])
    for fn in (lambda: oracle.attn_fwd(q, k, v, 0.5, sink=sg),
               lambda: oracle.attn_fwd_blockwise(q, k, v, 0.5, block=3, sink=sg)):
        o, lse = fn()
        assert np.all(np.isfinite(o)) and np.all(np.abs(o) < 1e-300)
        np.testing.assert_allclose(lse[0], np.broadcast_to(sg[:, None], (2, 5)), rtol=0, atol=1e-12)


@pytest.mark.parametrize("block", [1, 3, 64, 100])
@pytest.mark.parametrize("causal,window,n_sink", MODES)
def test_epilogue_sink_equals_extra_column(block, causal, window, n_sink):
    """The blockwise recurrence with the sink added once after the last block
    (ch.15 section 4.6's epilogue form) equals the two-pass definition with
    the sink as one more softmax column."""
    rng = np.random.default_rng(106)
    q, k, v = _rand(rng, 2, 11, 13, 4, 2, 8, qmul=2.0)
    sg = np.array([-np.inf, -2.0, 1.0, 25.0])
    o1, l1 = oracle.attn_fwd(q, k, v, 0.5, causal, window, n_sink, sink=sg)
    o2, l2 = oracle.attn_fwd_blockwise(q, k, v, 0.5, causal, window, n_sink, block=block, sink=sg)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-13)


@pytest.mark.parametrize("shape,causal,window,n_sink", [
    ((1, 5, 5, 2, 1, 4), False, 0, 0),
    ((1, 8, 5, 2, 2, 4), True, 0, 0),      # Sq > Skv: rows with no key
    ((2, 6, 8, 2, 1, 3), True, 2, 2),
])
def test_brute_force_with_sink(shape, causal, window, n_sink):
    """The C oracle with a sink equals the independent pure-Python brute force."""
    B, Sq, Skv, Hq, Hkv, d = shape
    rng = np.random.default_rng(107)
    q, k, v = _rand(rng, B, Sq, Skv, Hq, Hkv, d, qmul=2.0)
    sg = [0.9, -math.inf] if Hq == 2 else [0.9] * Hq
    o, lse = oracle.attn_fwd(q, k, v, 0.6, causal, window, n_sink, sink=sg)
    ob, lb = bf.attention(q.tolist(), k.tolist(), v.tolist(), 0.6, causal, window, n_sink, sink=sg)
    np.testing.assert_allclose(o, np.array(ob), rtol=0, atol=1e-13)
    lb = np.array(lb)
    assert np.array_equal(np.isneginf(lse), np.isneginf(lb))
    fin = np.isfinite(lb)
    np.testing.assert_allclose(lse[fin], lb[fin], rtol=0, atol=1e-13)


def test_varlen_and_decode_with_sink():
    """Varlen: each packed sequence equals its own dense call with the same
    sinks.  Decode: merging the sink-free split partials with the sink equals
    the one-row definition with the sink."""
    rng = np.random.default_rng(108)
    Hq, Hkv, d = 4, 2, 8
    sg = np.array([0.2, -np.inf, 3.0, -1.0])
    lens = [5, 1, 9]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    q = rng.normal(size=(T, Hq, d))
    k = rng.normal(size=(T, Hkv, d))
    v = rng.normal(size=(T, Hkv, d))
    o, lse = oracle.attn_fwd_varlen(q, k, v, cu, cu, 0.4, True, sink=sg)
    for s in range(len(lens)):
        a, b = cu[s], cu[s + 1]
        od, ld = oracle.attn_fwd(q[None, a:b], k[None, a:b], v[None, a:b], 0.4, True, sink=sg)
        np.testing.assert_array_equal(o[a:b], od[0])
        np.testing.assert_array_equal(lse[:, a:b], ld[0])
    B, Lmax = 3, 70
    L = [70, 0, 33]
    q = rng.normal(size=(B, Hq, d)) * 2
    k = rng.normal(size=(B, Lmax, Hkv, d))
    v = rng.normal(size=(B, Lmax, Hkv, d))
    od, ld = oracle.attn_decode(q, k, v, L, 0.35, sink=sg)
    op, lp = oracle.decode_split(q, k, v, L, 0.35, 4, page=16)
    oc, lc = oracle.combine(op, lp, sink=np.broadcast_to(sg, (B, Hq)))
    np.testing.assert_allclose(oc, od, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lc[np.isfinite(ld)], ld[np.isfinite(ld)], rtol=0, atol=1e-13)
    assert np.array_equal(np.isneginf(lc), np.isneginf(ld))
    # request 1 has no key: O = 0 and LSE = sigma (or -inf without a sink)
    assert np.all(od[1] == 0.0)
    np.testing.assert_array_equal(ld[1], sg)
