"""Tiny-shape brute force used to pin the oracle: pure Python scalars,
math.exp / math.fsum, key sets built explicitly.  Written independently of
oracle/attn_oracle.c (different structure: set of allowed keys first, then
exp of logits minus the max over that set, then a weighted sum)."""
import math


def allowed_keys(i, Sq, Skv, causal, window, n_sink):
    keys = set(range(Skv))
    if causal:
        shift = Skv - Sq                      # last query sees the last key
        keys = {j for j in keys if j - i <= shift}
        if window > 0:
            keys = {j for j in keys if (i + shift) - j < window or j < n_sink}
    return sorted(keys)


def attention(q, k, v, scale, causal=False, window=0, n_sink=0, sink=None):
    """q [B][Sq][Hq][d], k/v [B][Skv][Hkv][d] nested lists -> (o, lse) lists.
    sink: optional list of Hq logits, each a softmax column of its own whose
    value row is zero (None or -inf: no such column)."""
    B, Sq, Hq, d = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    Skv, Hkv = len(k[0]), len(k[0][0])
    G = Hq // Hkv
    o = [[[[0.0] * d for _ in range(Hq)] for _ in range(Sq)] for _ in range(B)]
    lse = [[[0.0] * Sq for _ in range(Hq)] for _ in range(B)]
    for b in range(B):
        for h in range(Hq):
            kh = h // G
            for i in range(Sq):
                keys = allowed_keys(i, Sq, Skv, causal, window, n_sink)
                extra = [] if sink is None or sink[h] == -math.inf else [sink[h]]
                if not keys and not extra:
                    lse[b][h][i] = -math.inf
                    continue
                logit = {j: scale * math.fsum(q[b][i][h][t] * k[b][j][kh][t] for t in range(d))
                         for j in keys}
                top = max(list(logit.values()) + extra)
                w = {j: math.exp(logit[j] - top) for j in keys}
                z = math.fsum(list(w.values()) + [math.exp(x - top) for x in extra])
                for t in range(d):
                    o[b][i][h][t] = math.fsum(w[j] * v[b][j][kh][t] for j in keys) / z
                lse[b][h][i] = top + math.log(z)
    return o, lse
