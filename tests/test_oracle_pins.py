"""Pins for the fp64 oracle: what the pages and the mathematics fix, checked
against the oracle on the CPU (no GPU).  Each pin is chosen so that a
plausible slip in the oracle (dropped scale, wrong sign of the max, strict
instead of inclusive causal diagonal, GQA index by modulo, transposed
operand, wrong LSE base, wrong split weights) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import _bruteforce as bf


def _np(t):
    return t.double().numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float64)


def _score_inputs(scores):
    """q, k, v such that scale * q.k_j == scores[j] exactly and V = identity:
    then O's row equals the softmax weights and LSE equals ln(sum exp)."""
    n = len(scores)
    d = n
    q = np.zeros((1, 1, 1, d))
    q[0, 0, 0, 0] = 1.0
    k = np.zeros((1, n, 1, d))
    k[0, :, 0, 0] = scores
    v = np.eye(n).reshape(1, n, 1, d)
    return q, k, v


# ---------------------------------------------------------------- worked examples

def test_worked_example_four_scores(gold):
    """llm-course ch.19 Flash Attention, section 19.5: scores [1,2,3,4]."""
    g = gold("softmax_four_scores.txt")
    q, k, v = _score_inputs(g["scores"])
    o, lse = oracle.attn_fwd(q, k, v, 1.0)
    assert np.round(o[0, 0, 0], 4).tolist() == g["weights"]
    assert round(math.exp(lse[0, 0, 0]), 2) == g["sum_exp"][0]
    # the same through the two-block online recurrence, with its running state
    o2, lse2, tr = oracle.attn_fwd_blockwise(q, k, v, 1.0, block=2, trace=True)
    assert np.round(o2[0, 0, 0], 4).tolist() == g["weights"]
    assert tr[0, 0] == g["block1_m"][0] and round(tr[0, 1], 4) == g["block1_l"][0]
    assert round(tr[0, 1] * math.exp(tr[0, 0] - tr[1, 0]), 4) == g["block1_l_rescaled"][0]
    assert tr[1, 0] == g["block2_m"][0] and round(tr[1, 1], 4) == g["block2_l"][0]


def test_worked_example_three_blocks(gold):
    """TileLang in practice: FlashAttention forward kernel, section 2.3:
    one score per block (1, 2, 3)."""
    g = gold("online_three_blocks.txt")
    q, k, v = _score_inputs(g["scores"])
    o, lse, tr = oracle.attn_fwd_blockwise(q, k, v, 1.0, block=1, trace=True)
    assert np.round(tr[:, 1], 3).tolist() == g["l"]
    # trace columns 2.. hold the unnormalised accumulator; V = I so column 2 is v1's coefficient
    assert np.round(tr[:, 2], 3).tolist() == g["v1_coeff"]
    alphas = [math.exp(tr[t - 1, 0] - tr[t, 0]) for t in (1, 2)]
    assert np.round(alphas, 3).tolist() == g["alpha"]
    assert np.round(o[0, 0, 0], 3).tolist() == g["weights"]
    o2, _ = oracle.attn_fwd(q, k, v, 1.0)
    assert np.round(o2[0, 0, 0], 3).tolist() == g["weights"]


def test_traffic_model_numbers(gold):
    """TileLang tutorial ch.15 section 1: the per-(b,h) element counts follow
    from the naive 4N^2 + 4Nd and fused Q + (N/Bm)(K + V) + O bookkeeping."""
    g = gold("traffic_model.txt")
    N, d, bm = (int(g[x][0]) for x in ("N", "d", "block_m"))
    assert 4 * N * N + 4 * N * d == g["naive_elements"][0]
    assert N * d * (2 + 2 * (N // bm)) == g["fused_elements"][0]
    assert 4 * N * N == g["sp_elements"][0]
    assert 4 * N * d == g["qkvo_elements"][0]


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("mode", ["full", "causal", "causal_sq_lt_skv", "window_sink"])
def test_zero_keys_give_uniform_mean(mode):
    """K = 0 makes every visible logit 0, so P is uniform over the visible
    keys: O is the mean of the visible V rows and LSE = ln(#visible)."""
    Sq, Skv, d = 9, 13, 4
    causal = mode != "full"
    window, n_sink = (3, 2) if mode == "window_sink" else (0, 0)
    if mode == "causal":
        Sq = Skv
    rng = np.random.default_rng(1)
    q = rng.normal(size=(1, Sq, 1, d))
    k = np.zeros((1, Skv, 1, d))
    v = rng.normal(size=(1, Skv, 1, d))
    o, lse = oracle.attn_fwd(q, k, v, 0.5, causal, window, n_sink)
    off = Skv - Sq
    for i in range(Sq):
        vis = [j for j in range(Skv)
               if (not causal or j <= i + off)
               and (window == 0 or j > i + off - window or j < n_sink)]
        np.testing.assert_allclose(o[0, i, 0], v[0, vis, 0].mean(0), rtol=0, atol=1e-13)
        assert abs(lse[0, 0, i] - math.log(len(vis))) < 1e-13


def test_single_key_and_causal_first_row():
    """One visible key: O = V_0 exactly and LSE = that key's logit.  Causal
    with Sq = Skv: row 0 sees only key 0."""
    rng = np.random.default_rng(2)
    d = 8
    q = rng.normal(size=(1, 1, 1, d))
    k = rng.normal(size=(1, 1, 1, d))
    v = rng.normal(size=(1, 1, 1, d))
    o, lse = oracle.attn_fwd(q, k, v, 0.3)
    assert np.array_equal(o[0, 0, 0], v[0, 0, 0])
    assert abs(lse[0, 0, 0] - 0.3 * float(q[0, 0, 0] @ k[0, 0, 0])) < 1e-14
    q = rng.normal(size=(2, 6, 3, d))
    k = rng.normal(size=(2, 6, 3, d))
    v = rng.normal(size=(2, 6, 3, d))
    o, _ = oracle.attn_fwd(q, k, v, 0.3, causal=True)
    assert np.array_equal(o[:, 0], v[:, 0])


def test_two_keys_logistic():
    """Two keys with logits a, b: weights are the logistic function of a - b."""
    d = 3
    q = np.array([1.0, 0.0, 0.0]).reshape(1, 1, 1, d)
    k = np.array([[0.7, 5.0, 1.0], [-1.9, 2.0, 3.0]]).reshape(1, 2, 1, d)
    v = np.array([[1.0, 2.0, -1.0], [4.0, -3.0, 0.5]]).reshape(1, 2, 1, d)
    s = 1.25
    a, b = s * 0.7, s * -1.9
    w0 = 1.0 / (1.0 + math.exp(b - a))
    o, lse = oracle.attn_fwd(q, k, v, s)
    np.testing.assert_allclose(o[0, 0, 0], w0 * v[0, 0, 0] + (1 - w0) * v[0, 1, 0], atol=1e-15)
    assert abs(lse[0, 0, 0] - math.log(math.exp(a) + math.exp(b))) < 1e-14


def test_fully_masked_rows_are_zero():
    """Causal with Sq > Skv (bottom-right aligned): the first Sq - Skv rows see
    no key: O = +0.0 exactly and LSE = -inf (ch.15 section 5.1(2))."""
    rng = np.random.default_rng(3)
    Sq, Skv = 11, 4
    q = rng.normal(size=(1, Sq, 2, 8))
    k = rng.normal(size=(1, Skv, 2, 8))
    v = rng.normal(size=(1, Skv, 2, 8))
    for fn in (lambda: oracle.attn_fwd(q, k, v, 0.4, True),
               lambda: oracle.attn_fwd_blockwise(q, k, v, 0.4, True, block=3)):
        o, lse = fn()
        assert np.all(o[0, : Sq - Skv] == 0.0) and not np.signbit(o[0, : Sq - Skv]).any()
        assert np.all(np.isneginf(lse[0, :, : Sq - Skv]))
        assert np.all(np.isfinite(lse[0, :, Sq - Skv:]))
        np.testing.assert_allclose(o[0, Sq - Skv], v[0, 0], atol=1e-15)  # sees key 0 only


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("causal,window,n_sink", [(False, 0, 0), (True, 0, 0), (True, 3, 1)])
def test_shift_invariance(causal, window, n_sink):
    """Adding one vector u to every key adds scale*(q_i . u) to all of row i's
    logits: O is unchanged and LSE_i moves by exactly that amount
    (ch.15 section 2.2; TileLang in practice section 2.1)."""
    rng = np.random.default_rng(4)
    B, Sq, Skv, H, d = 2, 7, 10, 2, 6
    q = rng.normal(size=(B, Sq, H, d))
    k = rng.normal(size=(B, Skv, H, d))
    v = rng.normal(size=(B, Skv, H, d))
    u = rng.normal(size=(d,)) * 3.0
    s = 0.37
    o1, l1 = oracle.attn_fwd(q, k, v, s, causal, window, n_sink)
    o2, l2 = oracle.attn_fwd(q, k + u, v, s, causal, window, n_sink)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    shift = s * np.einsum("bihd,d->bhi", q, u)
    fin = np.isfinite(l1)
    np.testing.assert_allclose((l2 - l1)[fin], shift[fin], rtol=0, atol=1e-12)


def test_rows_of_p_sum_to_one():
    """A constant value column c gives O = c in every row that sees a key."""
    rng = np.random.default_rng(5)
    q = rng.normal(size=(1, 12, 2, 4)) * 4
    k = rng.normal(size=(1, 12, 2, 4))
    v = rng.normal(size=(1, 12, 2, 4))
    v[..., 2] = 0.75
    for args in ((False, 0, 0), (True, 0, 0), (True, 4, 2)):
        o, _ = oracle.attn_fwd(q, k, v, 0.5, *args)
        np.testing.assert_allclose(o[..., 2], 0.75, rtol=0, atol=1e-14)


def test_mini_lab_tiled_equals_naive():
    """llm-course ch.19 section 19.12: Q/K/V of 16 x 8, tiles of 4, seed 0:
    tiled online softmax and the naive definition agree below 1e-12."""
    rng = np.random.default_rng(0)
    Q, K, V = (rng.normal(size=(16, 8)) for _ in range(3))
    q, k, v = (x.reshape(1, 16, 1, 8) for x in (Q, K, V))
    o1, _ = oracle.attn_fwd(q, k, v, 1 / math.sqrt(8))
    o2, _ = oracle.attn_fwd_blockwise(q, k, v, 1 / math.sqrt(8), block=4)
    assert np.abs(o1 - o2).max() < 1e-12


@pytest.mark.parametrize("block", [1, 3, 4, 64, 128, 100])
@pytest.mark.parametrize("mode", ["full", "causal", "causal_sq_ne_skv", "window_sink", "gqa"])
def test_blockwise_equals_two_pass(block, mode):
    """ch.15 section 2.4 (equivalence proof): the online recurrence returns the
    two-pass result for any block size, including 1 and non-divisors."""
    rng = np.random.default_rng(6)
    B, Sq, Skv, Hq, Hkv, d = 2, 37, 300, 2, 2, 16
    causal, window, n_sink = False, 0, 0
    if mode == "causal":
        causal, Sq = True, 300
    elif mode == "causal_sq_ne_skv":
        causal = True
    elif mode == "window_sink":
        causal, window, n_sink, Sq = True, 50, 3, 300
    elif mode == "gqa":
        Hq, causal = 4, True
    q = rng.normal(size=(B, Sq, Hq, d)) * 2
    k = rng.normal(size=(B, Skv, Hkv, d))
    v = rng.normal(size=(B, Skv, Hkv, d))
    o1, l1 = oracle.attn_fwd(q, k, v, 0.25, causal, window, n_sink)
    o2, l2 = oracle.attn_fwd_blockwise(q, k, v, 0.25, causal, window, n_sink, block=block)
    assert np.abs(o1 - o2).max() < 1e-12
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-12)


@pytest.mark.parametrize("shape,causal,window,n_sink", [
    ((1, 5, 5, 1, 1, 4), False, 0, 0),
    ((2, 4, 7, 2, 1, 3), False, 0, 0),
    ((1, 6, 6, 2, 2, 4), True, 0, 0),
    ((1, 8, 5, 2, 1, 4), True, 0, 0),      # Sq > Skv: masked rows
    ((1, 5, 8, 4, 2, 4), True, 0, 0),      # Sq < Skv: shifted diagonal
    ((1, 8, 8, 1, 1, 4), True, 3, 1),
    ((2, 6, 8, 2, 1, 2), True, 2, 2),
])
def test_brute_force_tiny(shape, causal, window, n_sink):
    """The C oracle equals an independently written pure-Python brute force."""
    B, Sq, Skv, Hq, Hkv, d = shape
    rng = np.random.default_rng(7)
    q = rng.normal(size=(B, Sq, Hq, d)) * 2
    k = rng.normal(size=(B, Skv, Hkv, d))
    v = rng.normal(size=(B, Skv, Hkv, d))
    o, lse = oracle.attn_fwd(q, k, v, 0.6, causal, window, n_sink)
    ob, lb = bf.attention(q.tolist(), k.tolist(), v.tolist(), 0.6, causal, window, n_sink)
    np.testing.assert_allclose(o, np.array(ob), rtol=0, atol=1e-13)
    lb = np.array(lb)
    assert np.array_equal(np.isneginf(lse), np.isneginf(lb))
    fin = np.isfinite(lb)
    np.testing.assert_allclose(lse[fin], lb[fin], rtol=0, atol=1e-13)


def test_bruteforce_itself_on_worked_example(gold):
    """The brute force reproduces the printed weights too (it is a pin only
    if it is right)."""
    g = gold("softmax_four_scores.txt")
    q, k, v = _score_inputs(g["scores"])
    o, _ = bf.attention(q.tolist(), k.tolist(), v.tolist(), 1.0)
    assert np.round(o[0][0][0], 4).tolist() == g["weights"]


# ---------------------------------------------------------------- structure: GQA, varlen, decode, split

def test_gqa_equals_mha_with_repeated_heads():
    """Query head h reads key/value head h // (Hq/Hkv) (ch.15 section 4.8(1)):
    GQA equals MHA on K/V whose heads are repeated group-wise."""
    rng = np.random.default_rng(8)
    B, S, Hq, Hkv, d = 2, 20, 8, 2, 8
    q = rng.normal(size=(B, S, Hq, d))
    k = rng.normal(size=(B, S, Hkv, d))
    v = rng.normal(size=(B, S, Hkv, d))
    o1, l1 = oracle.attn_fwd(q, k, v, 0.3, True)
    rep = np.repeat(np.arange(Hkv), Hq // Hkv)
    o2, l2 = oracle.attn_fwd(q, k[:, :, rep], v[:, :, rep], 0.3, True)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


@pytest.mark.parametrize("window,n_sink", [(0, 0), (5, 1)])
def test_varlen_equals_per_sequence(window, n_sink):
    """Packed sequences with cu_seqlens (ch.15 section 5.3) equal separate
    dense calls, each right-aligned (off = Lk - Lq)."""
    rng = np.random.default_rng(9)
    lq, lk = [5, 1, 17, 9], [5, 3, 17, 20]
    Hq, Hkv, d = 4, 2, 8
    cu_q, cu_k = np.cumsum([0] + lq), np.cumsum([0] + lk)
    q = rng.normal(size=(cu_q[-1], Hq, d))
    k = rng.normal(size=(cu_k[-1], Hkv, d))
    v = rng.normal(size=(cu_k[-1], Hkv, d))
    o, lse = oracle.attn_fwd_varlen(q, k, v, cu_q, cu_k, 0.4, True, window, n_sink)
    for s in range(len(lq)):
        a, e, ka, ke = cu_q[s], cu_q[s + 1], cu_k[s], cu_k[s + 1]
        od, ld = oracle.attn_fwd(q[None, a:e], k[None, ka:ke], v[None, ka:ke], 0.4, True,
                                 window, n_sink)
        np.testing.assert_array_equal(o[a:e], od[0])
        np.testing.assert_array_equal(lse[:, a:e], ld[0])


def test_decode_equals_one_row_forward():
    """Decode of request b is a one-row forward over its first L_b keys."""
    rng = np.random.default_rng(10)
    B, Hq, Hkv, d, Lmax = 3, 4, 2, 8, 40
    L = [40, 1, 23]
    q = rng.normal(size=(B, Hq, d))
    k = rng.normal(size=(B, Lmax, Hkv, d))
    v = rng.normal(size=(B, Lmax, Hkv, d))
    o, lse = oracle.attn_decode(q, k, v, L, 0.35)
    for b in range(B):
        od, ld = oracle.attn_fwd(q[b][None, None], k[b:b + 1, : L[b]], v[b:b + 1, : L[b]], 0.35)
        np.testing.assert_array_equal(o[b], od[0, 0])
        np.testing.assert_array_equal(lse[b], ld[0, :, 0])


@pytest.mark.parametrize("num_splits", [1, 2, 3, 8, 40])
def test_split_combine_equals_unsplit(num_splits):
    """ch.15 section 5.4: merging split partials with weights exp(lse_s - M)
    gives the unsplit result for any partition, including empty splits."""
    rng = np.random.default_rng(11)
    B, Hq, Hkv, d, Lmax = 4, 4, 2, 8, 200
    L = [200, 17, 1, 129]
    q = rng.normal(size=(B, Hq, d)) * 3
    k = rng.normal(size=(B, Lmax, Hkv, d))
    v = rng.normal(size=(B, Lmax, Hkv, d))
    o, lse = oracle.attn_decode(q, k, v, L, 0.35)
    op, lp = oracle.decode_split(q, k, v, L, 0.35, num_splits, page=16)
    oc, lc = oracle.combine(op, lp)
    np.testing.assert_allclose(oc, o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lc, lse, rtol=0, atol=1e-13)
    # splits beyond a request's page count are empty: weight 0, lse -inf
    npages = [(x + 15) // 16 for x in L]
    for b in range(B):
        pps = -(-npages[b] // num_splits)
        for s in range(num_splits):
            assert np.isneginf(lp[b, :, s]).all() == (s * pps >= npages[b])


def test_combine_weights_are_l_fractions():
    """The merge weight of split s is l_s / sum l (ch.15 section 5.4): two
    splits with equal lse get equal weight, whatever their outputs."""
    op = np.array([[[1.0, 0.0], [0.0, 1.0]]])          # [rows=1, S=2, d=2]
    lp = np.array([[math.log(3.0), math.log(3.0)]])
    o, lse = oracle.combine(op, lp)
    np.testing.assert_allclose(o, [[0.5, 0.5]], atol=1e-15)
    assert abs(lse[0] - math.log(6.0)) < 1e-15
    lp = np.array([[math.log(1.0), math.log(3.0)]])
    o, _ = oracle.combine(op, lp)
    np.testing.assert_allclose(o, [[0.25, 0.75]], atol=1e-15)


def test_oracle_on_paged_generator_matches_contiguous_layout():
    """The generator's page scatter keeps each request's tokens in order:
    gathering them back through the page table gives the contiguous caches."""
    x = workloads.paged_decode_inputs(77, 5, 4, 2, 16, 1, 70, page=16)
    k, v = x.contiguous_kv(list(range(5)))
    for b in range(5):
        L = int(x.seqlens[b])
        pages = x.page_table[b, : (L + 15) // 16].long()
        kk = x.k_pages[pages].reshape(-1, 2, 16)[:L]
        vv = x.v_pages[pages].reshape(-1, 2, 16)[:L]
        assert torch.equal(kk, k[b, :L]) and torch.equal(vv, v[b, :L])
    assert int((x.page_table >= 0).sum()) == sum((int(L) + 15) // 16 for L in x.seqlens)


def test_bf16_inputs_are_exact_in_fp64():
    """The oracle sees the bf16 values exactly: the fp64 upcast of a bf16
    tensor round-trips."""
    x = workloads.dense_inputs(5, 1, 2, 2, 8, 8, 16, q_mult=8.0)
    assert torch.equal(x.q.double().to(torch.bfloat16), x.q)
    q32 = torch.randn(4, generator=torch.Generator().manual_seed(1)) * 8
    assert torch.equal((q32.to(torch.bfloat16).double() * 1).to(torch.bfloat16), q32.to(torch.bfloat16))
