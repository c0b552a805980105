"""Pins for the oracle's backward pass: central finite differences of the
forward oracle (an independent route to the same gradients), the zero sum of
dK over a key head (the forward is invariant to a common shift of all keys),
a closed form for dV with uniform probabilities, and GQA as repeated heads.
A plausible slip (missing D term, wrong scale placement, dK taken from dS
instead of its transpose, GQA accumulation to the wrong head) fails one."""
import numpy as np
import pytest

import oracle

MODES = [(False, 0, 0), (True, 0, 0), (True, 2, 1)]


def _loss_grad_fd(q, k, v, g, scale, causal, window, n_sink, which, h=1e-6):
    args = {"q": q, "k": k, "v": v}
    x = args[which]
    num = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp = x.copy(); xp[idx] += h
        xm = x.copy(); xm[idx] -= h
        a = dict(args, **{which: xp}); b = dict(args, **{which: xm})
        op, _ = oracle.attn_fwd(a["q"], a["k"], a["v"], scale, causal, window, n_sink)
        om, _ = oracle.attn_fwd(b["q"], b["k"], b["v"], scale, causal, window, n_sink)
        num[idx] = ((op - om) * g).sum() / (2 * h)
    return num


@pytest.mark.parametrize("causal,window,n_sink", MODES)
@pytest.mark.parametrize("shape", [(1, 3, 4, 2, 1, 3), (2, 4, 3, 2, 2, 2), (1, 5, 5, 3, 1, 2)])
def test_finite_differences(shape, causal, window, n_sink):
    B, Sq, Skv, Hq, Hkv, d = shape
    rng = np.random.default_rng(sum(shape) + 10 * causal + window)
    q = rng.normal(size=(B, Sq, Hq, d))
    k = rng.normal(size=(B, Skv, Hkv, d))
    v = rng.normal(size=(B, Skv, Hkv, d))
    g = rng.normal(size=(B, Sq, Hq, d))
    dq, dk, dv = oracle.attn_bwd(q, k, v, g, 0.7, causal, window, n_sink)
    for name, an in (("q", dq), ("k", dk), ("v", dv)):
        num = _loss_grad_fd(q, k, v, g, 0.7, causal, window, n_sink, name)
        np.testing.assert_allclose(an, num, rtol=0, atol=2e-8, err_msg=name)


@pytest.mark.parametrize("causal,window,n_sink", MODES)
def test_dk_sums_to_zero(causal, window, n_sink):
    """Adding one vector to every key moves all visible logits of a row by the
    same amount, leaving O unchanged: the key gradients of a head sum to 0."""
    rng = np.random.default_rng(21)
    q = rng.normal(size=(2, 9, 4, 8)) * 2
    k = rng.normal(size=(2, 11, 2, 8))
    v = rng.normal(size=(2, 11, 2, 8))
    g = rng.normal(size=(2, 9, 4, 8))
    _, dk, _ = oracle.attn_bwd(q, k, v, g, 0.5, causal, window, n_sink)
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)


def test_uniform_probabilities_closed_form():
    """K = 0: each row's probabilities are 1/n over its n visible keys, so
    dV_j = sum over the rows i that see j of dO_i / n_i, and dQ = 0."""
    rng = np.random.default_rng(22)
    Sq = Skv = 7
    q = rng.normal(size=(1, Sq, 1, 4))
    k = np.zeros((1, Skv, 1, 4))
    v = rng.normal(size=(1, Skv, 1, 4))
    g = rng.normal(size=(1, Sq, 1, 4))
    dq, _, dv = oracle.attn_bwd(q, k, v, g, 0.5, causal=True)
    exp = np.zeros((Skv, 4))
    for i in range(Sq):
        for j in range(i + 1):
            exp[j] += g[0, i, 0] / (i + 1)
    np.testing.assert_allclose(dv[0, :, 0], exp, atol=1e-14)
    np.testing.assert_allclose(dq, 0.0, atol=1e-14)


def test_gqa_equals_summed_mha():
    """With Hq/Hkv query heads per key head, dK and dV of the shared head are
    the sums of the per-query-head gradients of the repeated-head MHA."""
    rng = np.random.default_rng(23)
    q = rng.normal(size=(1, 6, 4, 8))
    k = rng.normal(size=(1, 9, 2, 8))
    v = rng.normal(size=(1, 9, 2, 8))
    g = rng.normal(size=(1, 6, 4, 8))
    dq, dk, dv = oracle.attn_bwd(q, k, v, g, 0.4, causal=True)
    kr, vr = np.repeat(k, 2, axis=2), np.repeat(v, 2, axis=2)
    dq2, dk2, dv2 = oracle.attn_bwd(q, kr, vr, g, 0.4, causal=True)
    np.testing.assert_allclose(dq, dq2, atol=1e-13)
    np.testing.assert_allclose(dk, dk2.reshape(1, 9, 2, 2, 8).sum(3), atol=1e-13)
    np.testing.assert_allclose(dv, dv2.reshape(1, 9, 2, 2, 8).sum(3), atol=1e-13)


# ------------------------------------------------------------------ logit sink

def _sink_fd(q, k, v, g, scale, causal, window, n_sink, sink, which, h=1e-6):
    """Central differences of sum(O * g) for the forward with a logit sink,
    with respect to q, k, v or the sink vector."""
    args = {"q": q, "k": k, "v": v, "sink": sink}
    x = args[which]
    num = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp = x.copy(); xp[idx] += h
        xm = x.copy(); xm[idx] -= h
        a = dict(args, **{which: xp}); b = dict(args, **{which: xm})
        op, _ = oracle.attn_fwd(a["q"], a["k"], a["v"], scale, causal, window, n_sink,
                                sink=a["sink"])
        om, _ = oracle.attn_fwd(b["q"], b["k"], b["v"], scale, causal, window, n_sink,
                                sink=b["sink"])
        num[idx] = ((op - om) * g).sum() / (2 * h)
    return num


@pytest.mark.parametrize("causal,window,n_sink", MODES)
@pytest.mark.parametrize("shape", [(1, 3, 4, 2, 1, 3), (2, 4, 3, 4, 2, 2)])
def test_sink_finite_differences(shape, causal, window, n_sink):
    """The logit sink's backward against central differences of the forward
    oracle with the sink: dq, dk, dv and the sink's own gradient."""
    B, Sq, Skv, Hq, Hkv, d = shape
    rng = np.random.default_rng(sum(shape) + 7 * causal + window + 100)
    q = rng.normal(size=(B, Sq, Hq, d))
    k = rng.normal(size=(B, Skv, Hkv, d))
    v = rng.normal(size=(B, Skv, Hkv, d))
    g = rng.normal(size=(B, Sq, Hq, d))
    sink = rng.normal(size=Hq)
    dq, dk, dv, ds = oracle.attn_bwd(q, k, v, g, 0.7, causal, window, n_sink, sink=sink)
    for name, an in (("q", dq), ("k", dk), ("v", dv), ("sink", ds)):
        num = _sink_fd(q, k, v, g, 0.7, causal, window, n_sink, sink, name)
        np.testing.assert_allclose(an, num, rtol=0, atol=2e-8, err_msg=name)


def test_sink_minus_inf_is_no_sink():
    """A sink of -inf for every head gives the sink-free gradients bit for bit
    and a zero sink gradient."""
    rng = np.random.default_rng(31)
    q = rng.normal(size=(2, 6, 4, 3))
    k = rng.normal(size=(2, 7, 2, 3))
    v = rng.normal(size=(2, 7, 2, 3))
    g = rng.normal(size=(2, 6, 4, 3))
    ref = oracle.attn_bwd(q, k, v, g, 0.6, True)
    got = oracle.attn_bwd(q, k, v, g, 0.6, True, sink=np.full(4, -np.inf))
    for a, b in zip(ref, got[:3]):
        assert np.array_equal(a, b)
    assert np.array_equal(got[3], np.zeros(4))


def test_sink_gradient_one_key_closed_form():
    """One key: O = P v with P = logistic(s - sigma); dL/dsigma = -P (1 - P) g.v."""
    rng = np.random.default_rng(32)
    q = rng.normal(size=(1, 1, 1, 3))
    k = rng.normal(size=(1, 1, 1, 3))
    v = rng.normal(size=(1, 1, 1, 3))
    g = rng.normal(size=(1, 1, 1, 3))
    sg = np.array([0.4])
    s = 0.9 * float(q.ravel() @ k.ravel())
    P = 1.0 / (1.0 + np.exp(sg[0] - s))
    *_, ds = oracle.attn_bwd(q, k, v, g, 0.9, False, sink=sg)
    assert np.isclose(ds[0], -P * (1 - P) * float(g.ravel() @ v.ravel()), rtol=1e-12, atol=0)
