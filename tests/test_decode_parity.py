"""GPU parity of the paged split-KV decode (attn_decode_paged through the C ABI)
against the fp64 oracle, which reads the same tokens from contiguous caches."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._parity import assert_masked_rows_zero, compare, np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ea():
    import exact_attention_08_gb300 as m
    assert torch.cuda.is_available()
    return m


def run_decode(ea, x, num_splits=None, workspace=None):
    o, lse = ea.attn_decode_paged(x.q.cuda(), x.k_pages.cuda(), x.v_pages.cuda(),
                                  x.page_table.cuda(), x.seqlens.cuda(),
                                  num_splits=num_splits or x.num_splits, scale=x.scale,
                                  workspace=workspace)
    torch.cuda.synchronize()
    return o, lse


def oracle_decode(x, requests):
    k, v = x.contiguous_kv(requests)
    return oracle.attn_decode(np64(x.q[requests]), np64(k), np64(v),
                              x.seqlens[requests].numpy(), x.scale)


@pytest.mark.parametrize("Hq,Hkv,d,splits", [
    (8, 2, 128, 1), (8, 2, 128, 3), (8, 2, 128, 8), (32, 8, 128, 8),
    (4, 4, 128, 5), (8, 1, 64, 8), (64, 2, 128, 4), (16, 16, 64, 2),
    (64, 1, 128, 3),  # 64 query heads on one KV head: four head chunks
])
def test_small(ea, Hq, Hkv, d, splits):
    lengths = [1, 15, 16, 17, 300, 0, 64, 1000]
    x = workloads.paged_decode_inputs(51, len(lengths), Hq, Hkv, d, 0, 0, lengths=lengths,
                                      num_splits=splits, extra_pages=7)
    o, lse = run_decode(ea, x)
    assert ea.attn_device_status() == ea.ATTN_OK
    ro, rl = oracle_decode(x, list(range(len(lengths))))
    compare(o, lse, ro, rl, f"decode Hq={Hq} Hkv={Hkv} d={d} S={splits}")
    assert_masked_rows_zero(o, np.isneginf(rl), "decode empty request")


def test_more_splits_than_pages(ea):
    x = workloads.paged_decode_inputs(52, 3, 8, 2, 128, 0, 0, lengths=[20, 3, 48], num_splits=16)
    o, lse = run_decode(ea, x)
    assert ea.attn_device_status() == ea.ATTN_OK
    ro, rl = oracle_decode(x, [0, 1, 2])
    compare(o, lse, ro, rl, "splits > pages")


def test_deterministic(ea):
    x = workloads.paged_decode_inputs(53, 6, 32, 8, 128, 100, 3000, num_splits=8)
    o1, l1 = run_decode(ea, x)
    o2, l2 = run_decode(ea, x)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


def test_bad_page_index_is_reported(ea):
    x = workloads.paged_decode_inputs(54, 2, 8, 2, 128, 0, 0, lengths=[40, 40], num_splits=2)
    pt = x.page_table.clone()
    pt[1, 1] = x.k_pages.shape[0] + 5  # past the pool: the kernel must not read it
    o, lse = ea.attn_decode_paged(x.q.cuda(), x.k_pages.cuda(), x.v_pages.cuda(), pt.cuda(),
                                  x.seqlens.cuda(), num_splits=2, scale=x.scale)
    assert ea.attn_device_status() == ea.ATTN_ERR_BAD_INPUT
    assert ea.attn_device_status() == ea.ATTN_OK  # cleared
    ro, rl = oracle_decode(x, [0])                 # request 0 is untouched
    compare(o[:1], lse[:1], ro, rl, "good request next to a bad one")


def test_many_short_requests(ea):
    """512 requests of 1-64 tokens: the request order's buckets hold many
    requests each, and most splits of a request are empty."""
    x = workloads.paged_decode_inputs(5802, 512, 32, 8, 128, 1, 64, num_splits=8)
    o, lse = run_decode(ea, x)
    assert ea.attn_device_status() == ea.ATTN_OK
    ro, rl = oracle_decode(x, list(range(512)))
    compare(o, lse, ro, rl, "many short requests")


def test_long_requests(ea):
    """Requests of 30,000-65,536 tokens (about 2,000-4,100 pages each, 8
    splits of about 250-500 pages) through the workspace decode."""
    x = workloads.paged_decode_inputs(5801, 4, 32, 8, 128, 30000, 65536, num_splits=8)
    o, lse = run_decode(ea, x)
    assert ea.attn_device_status() == ea.ATTN_OK
    ro, rl = oracle_decode(x, list(range(4)))
    e = compare(o, lse, ro, rl, "long requests")
    print("decode long requests errors", e)


def test_full_size(ea):
    x = workloads.paged_decode()
    ws = torch.empty(ea.attn_decode_workspace_size(64, 32, 128, 8), dtype=torch.uint8,
                     device="cuda")
    o, lse = run_decode(ea, x, workspace=ws)
    assert ea.attn_device_status() == ea.ATTN_OK
    worst = (0.0, 0.0)
    for c in range(0, 64, 8):
        req = list(range(c, c + 8))
        ro, rl = oracle_decode(x, req)
        e = compare(o[c:c + 8], lse[c:c + 8], ro, rl, f"decode requests {c}..{c + 7}")
        worst = tuple(max(a, b) for a, b in zip(worst, e))
    print("decode full size errors", worst)
