"""Seeded synthetic inputs for the exact-attention workloads.

This module is the ONLY code shared by the CUDA path's callers (tests, bench)
and the CPU oracle.  It draws random tensors and builds index structures
(sequence offsets, page tables); it holds none of the attention arithmetic.

Recipe (the same for every workload):
  * ``torch.Generator('cpu').manual_seed(seed)``; draws happen in a fixed
    order (lengths first, then q, k, v, then page permutation / padding);
  * values are fp32 ``randn`` (iid N(0,1)) cast to bf16; the oracle receives
    these bf16 values upcast exactly to fp64, never the fp32 draws;
  * seeds are ``config_index * 1000 + variant_index``.

Workload shapes are those of the five configurations the attention kernels
are measured on (tiny MHA, prefill MHA, long causal / sliding window with a
sink token, GQA causal / varlen, paged decode).  No public dataset is
involved: every input is synthetic.
"""
from __future__ import annotations

from dataclasses import dataclass, field
import math

import torch


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _randn_bf16(g: torch.Generator, shape, mult: float = 1.0) -> torch.Tensor:
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if mult != 1.0:
        x = x * mult
    return x.to(torch.bfloat16)


@dataclass
class DenseInputs:
    """Dense BSHD inputs: q [B,Sq,Hq,d], k/v [B,Skv,Hkv,d] (bf16, CPU)."""
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    causal: bool
    window: int
    n_sink: int
    scale: float
    seed: int

    @property
    def shape(self):
        B, Sq, Hq, d = self.q.shape
        return B, Hq, self.k.shape[2], Sq, self.k.shape[1], d


def dense_inputs(seed: int, B: int, Hq: int, Hkv: int, Sq: int, Skv: int, d: int,
                 causal: bool = False, window: int = 0, n_sink: int = 0,
                 q_mult: float = 1.0, scale: float | None = None) -> DenseInputs:
    """iid N(0,1) bf16 Q/K/V; ``q_mult`` multiplies Q before the bf16 cast
    (a power of two keeps the cast exact: the x8 softmax stress variant)."""
    g = _gen(seed)
    q = _randn_bf16(g, (B, Sq, Hq, d), q_mult)
    k = _randn_bf16(g, (B, Skv, Hkv, d))
    v = _randn_bf16(g, (B, Skv, Hkv, d))
    return DenseInputs(q, k, v, causal, window, n_sink,
                       scale if scale is not None else 1.0 / math.sqrt(d), seed)


@dataclass
class VarlenInputs:
    """Packed inputs: q [Tq,Hq,d], k/v [Tk,Hkv,d], cu_seqlens int32 [nseq+1]."""
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    cu_q: torch.Tensor
    cu_k: torch.Tensor
    max_q: int
    max_k: int
    causal: bool
    window: int
    n_sink: int
    scale: float
    seed: int


def varlen_inputs(seed: int, nseq: int, lo: int, hi: int, Hq: int, Hkv: int, d: int,
                  causal: bool = True, window: int = 0, n_sink: int = 0,
                  lengths: list[int] | None = None, klengths: list[int] | None = None
                  ) -> VarlenInputs:
    """Self-attention packing: lengths uniform in [lo, hi] (inclusive) drawn from
    the seed unless given; key lengths equal query lengths unless given."""
    g = _gen(seed)
    if lengths is None:
        lengths = torch.randint(lo, hi + 1, (nseq,), generator=g).tolist()
    if klengths is None:
        klengths = list(lengths)
    cu_q = torch.tensor([0] + list(_cumsum(lengths)), dtype=torch.int32)
    cu_k = torch.tensor([0] + list(_cumsum(klengths)), dtype=torch.int32)
    Tq, Tk = int(cu_q[-1]), int(cu_k[-1])
    q = _randn_bf16(g, (Tq, Hq, d))
    k = _randn_bf16(g, (Tk, Hkv, d))
    v = _randn_bf16(g, (Tk, Hkv, d))
    return VarlenInputs(q, k, v, cu_q, cu_k, max(lengths) if lengths else 0,
                        max(klengths) if klengths else 0, causal, window, n_sink,
                        1.0 / math.sqrt(d), seed)


def _cumsum(xs):
    s = 0
    for x in xs:
        s += int(x)
        yield s


@dataclass
class PagedDecodeInputs:
    """One-token decode over a paged KV cache.

    q [B,Hq,d]; per-request keys/values packed token-major in k_flat/v_flat
    [sum L, Hkv, d] with offsets cu_kv [B+1]; the same tokens scattered into
    the page pools k_pages/v_pages [num_pages, page, Hkv, d] through
    page_table [B, max_pages] (int32, -1 past each request's last page).
    Slots past L_b in a request's last page hold junk (large keys) so that a
    missing length mask shows up as a wrong answer.
    """
    q: torch.Tensor
    k_flat: torch.Tensor
    v_flat: torch.Tensor
    cu_kv: torch.Tensor
    seqlens: torch.Tensor
    k_pages: torch.Tensor
    v_pages: torch.Tensor
    page_table: torch.Tensor
    page: int
    num_splits: int
    scale: float
    seed: int
    extra: dict = field(default_factory=dict)

    def contiguous_kv(self, requests):
        """k, v [len(requests), Lmax, Hkv, d] (zero padded) for the oracle."""
        L = [int(self.seqlens[b]) for b in requests]
        Lmax = max(L) if L else 0
        Hkv, d = self.k_flat.shape[1], self.k_flat.shape[2]
        k = torch.zeros(len(requests), Lmax, Hkv, d, dtype=self.k_flat.dtype)
        v = torch.zeros_like(k)
        for r, b in enumerate(requests):
            a, e = int(self.cu_kv[b]), int(self.cu_kv[b + 1])
            k[r, : e - a] = self.k_flat[a:e]
            v[r, : e - a] = self.v_flat[a:e]
        return k, v


def paged_decode_inputs(seed: int, B: int, Hq: int, Hkv: int, d: int, lo: int, hi: int,
                        page: int = 16, num_splits: int = 8,
                        lengths: list[int] | None = None, extra_pages: int = 0
                        ) -> PagedDecodeInputs:
    """Lengths uniform in [lo, hi] (inclusive) unless given; physical pages are
    a seeded random permutation of 0..num_pages-1 (plus ``extra_pages`` unused
    pages so the pool is not exactly full)."""
    g = _gen(seed)
    if lengths is None:
        lengths = torch.randint(lo, hi + 1, (B,), generator=g).tolist()
    seqlens = torch.tensor(lengths, dtype=torch.int32)
    cu = torch.tensor([0] + list(_cumsum(lengths)), dtype=torch.int64)
    T = int(cu[-1])
    q = _randn_bf16(g, (B, Hq, d))
    k_flat = _randn_bf16(g, (T, Hkv, d))
    v_flat = _randn_bf16(g, (T, Hkv, d))
    npages = [(L + page - 1) // page for L in lengths]
    total_pages = sum(npages) + extra_pages
    max_pages = max(npages) if npages else 0
    perm = torch.randperm(total_pages, generator=g).to(torch.int32)
    page_table = torch.full((B, max(max_pages, 1)), -1, dtype=torch.int32)
    k_pages = torch.zeros(max(total_pages, 1), page, Hkv, d, dtype=torch.bfloat16)
    v_pages = torch.zeros_like(k_pages)
    nxt = 0
    for b, L in enumerate(lengths):
        n = npages[b]
        phys = perm[nxt: nxt + n]
        nxt += n
        page_table[b, :n] = phys
        if n == 0:
            continue
        a = int(cu[b])
        full = L // page
        if full:
            k_pages[phys[:full].long()] = k_flat[a: a + full * page].view(full, page, Hkv, d)
            v_pages[phys[:full].long()] = v_flat[a: a + full * page].view(full, page, Hkv, d)
        rem = L - full * page
        if rem:
            pl = int(phys[full])
            k_pages[pl, :rem] = k_flat[a + full * page: a + L]
            v_pages[pl, :rem] = v_flat[a + full * page: a + L]
    # junk in the unused slots of every last page and in the unused pages
    used = torch.zeros(k_pages.shape[0], page, dtype=torch.bool)
    for b, L in enumerate(lengths):
        n = npages[b]
        if n:
            used[page_table[b, :n].long()] = True
            rem = L - (n - 1) * page
            used[int(page_table[b, n - 1]), rem:] = False
    n_free = int((~used).sum())
    k_pages[~used] = _randn_bf16(g, (n_free, Hkv, d), 16.0)
    v_pages[~used] = _randn_bf16(g, (n_free, Hkv, d))
    return PagedDecodeInputs(q, k_flat, v_flat, cu, seqlens, k_pages, v_pages, page_table, page,
                             num_splits, 1.0 / math.sqrt(d), seed)


@dataclass
class PagedPrefillInputs:
    """Packed queries q [Tq,Hq,d] with cu_q [B+1] against the paged cache of
    ``cache`` (its k_flat/v_flat [Tk,Hkv,d] with cu_kv [B+1] are the same keys
    contiguously, for the oracle)."""
    q: torch.Tensor
    cu_q: torch.Tensor
    max_q: int
    cache: "PagedDecodeInputs"
    scale: float
    seed: int


def paged_prefill_inputs(seed: int, B: int, Hq: int, Hkv: int, d: int, lk_lo: int, lk_hi: int,
                         lq_lo: int, lq_hi: int, lengths_k: list[int] | None = None,
                         lengths_q: list[int] | None = None) -> PagedPrefillInputs:
    """A paged cache as for decode (key counts uniform in [lk_lo, lk_hi] unless
    given, pages in a seeded random permutation, junk in unused slots), then
    per sequence a block of query rows, lengths uniform in [lq_lo, lq_hi]
    unless given, drawn from a second generator seeded seed + 500."""
    cache = paged_decode_inputs(seed, B, Hq, Hkv, d, lk_lo, lk_hi, lengths=lengths_k)
    g = _gen(seed + 500)
    if lengths_q is None:
        lengths_q = torch.randint(lq_lo, lq_hi + 1, (B,), generator=g).tolist()
    cu_q = torch.tensor([0] + list(_cumsum(lengths_q)), dtype=torch.int32)
    q = _randn_bf16(g, (int(cu_q[-1]), Hq, d))
    return PagedPrefillInputs(q, cu_q, max(lengths_q) if lengths_q else 0, cache,
                              1.0 / math.sqrt(d), seed)


def chunked_prefill():
    """Chunked prefill on a paged cache: B=8, Hq=32, Hkv=8, d=128, cache lengths
    uniform in [2048, 8192], the last 512 tokens of each as the query block."""
    return paged_prefill_inputs(6001, 8, 32, 8, 128, 2048, 8192, 512, 512)


def grad_output(seed: int, shape) -> torch.Tensor:
    """A seeded output gradient dO for the backward pass: iid N(0,1) cast to bf16."""
    return _randn_bf16(_gen(seed), tuple(shape))


def logit_sinks(seed: int, Hq: int, lo: float = 4.0, hi: float = 12.0,
                extremes: bool = False) -> torch.Tensor:
    """Per-head logit sinks [Hq] fp32 (CPU), uniform in [lo, hi]: around the
    log-sum-exp of a row of a few thousand N(0,1)-scaled scores, so the sink
    takes anything from a few percent to nearly all of each row's weight.
    extremes: head 0 gets -inf (no sink), head 1 (if any) +100 (e^100
    overflows fp32: the sink dominates), head 2 (if any) -30 (negligible)."""
    g = _gen(seed)
    s = lo + (hi - lo) * torch.rand(Hq, generator=g, dtype=torch.float32)
    if extremes:
        for h, val in enumerate((-math.inf, 100.0, -30.0)):
            if h < Hq:
                s[h] = val
    return s


# --------------------------------------------------------------------------
# The measured workloads, by name.  Each entry builds its inputs from a seed.
# --------------------------------------------------------------------------

def tiny_mha():
    """B=1, H=1, Sq=Skv=128, d=64, non-causal."""
    return dense_inputs(1001, 1, 1, 1, 128, 128, 64)


def prefill_mha(causal: bool, stress: bool = False):
    """B=4, H=16, Sq=Skv=2048, d=128; stress multiplies Q by 8."""
    variant = 1 + int(causal) + 2 * int(stress)
    return dense_inputs(2000 + variant, 4, 16, 16, 2048, 2048, 128, causal=causal,
                        q_mult=8.0 if stress else 1.0)


def long_causal(window: bool = False):
    """B=1, H=16, S=8192, d=128 causal; window variant: W=1024 keys plus the
    token at position 0 always visible (one sink key)."""
    if window:
        return dense_inputs(3002, 1, 16, 16, 8192, 8192, 128, causal=True, window=1024, n_sink=1)
    return dense_inputs(3001, 1, 16, 16, 8192, 8192, 128, causal=True)


def gqa_causal():
    """B=2, Hq=32, Hkv=8, S=4096, d=128, causal."""
    return dense_inputs(4001, 2, 32, 8, 4096, 4096, 128, causal=True)


def gqa_varlen():
    """8 packed sequences, lengths uniform in [256, 4096], Hq=32, Hkv=8, d=128, causal."""
    return varlen_inputs(4002, 8, 256, 4096, 32, 8, 128, causal=True)


def paged_decode():
    """B=64, Hq=32, Hkv=8, d=128, L uniform in [1024, 8192], 16-token pages, 8 splits."""
    return paged_decode_inputs(5001, 64, 32, 8, 128, 1024, 8192, page=16, num_splits=8)
