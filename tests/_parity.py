"""Comparison helpers for the GPU parity tests (CUDA path vs the fp64 oracle).

Tolerances: O within 1e-2 absolute of the oracle's fp64 value, plus half a
bf16 unit in the last place of that value (the output is bf16: above 4 the
format itself cannot come within 1e-2, so the bound is read as applying to
the value before its final rounding); LSE within 1e-3 absolute.  Rows that
see no key must be exactly +0.0 in O and -inf in LSE.
"""
import numpy as np
import torch

O_TOL = 1e-2
LSE_TOL = 1e-3


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    a = np.abs(x)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 0.5 * np.exp2(e - 7)


def compare(o_gpu: torch.Tensor, lse_gpu: torch.Tensor, o_ref: np.ndarray, lse_ref: np.ndarray,
            what: str = ""):
    """o_gpu/o_ref share a layout with the row axis aligned; lse likewise.
    Returns (max_abs_err_o, max_abs_err_lse) over rows that see keys."""
    og = o_gpu.float().cpu().numpy().astype(np.float64)
    lg = lse_gpu.float().cpu().numpy().astype(np.float64)
    assert og.shape == o_ref.shape, (og.shape, o_ref.shape)
    assert lg.shape == lse_ref.shape, (lg.shape, lse_ref.shape)
    assert np.all(np.isfinite(og)), f"{what}: non-finite O"
    masked = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lg), masked), f"{what}: -inf LSE pattern differs"
    fin = ~masked
    err_l = float(np.abs(lg[fin] - lse_ref[fin]).max()) if fin.any() else 0.0
    assert err_l <= LSE_TOL, f"{what}: LSE error {err_l:.3e}"
    diff = np.abs(og - o_ref)
    bound = O_TOL + bf16_half_ulp(o_ref)
    bad = diff > bound
    assert not bad.any(), (f"{what}: O error {diff.max():.3e} at {np.unravel_index(diff.argmax(), diff.shape)}"
                           f" ({int(bad.sum())} elements over bound)")
    return float(diff.max()), err_l


def assert_masked_rows_zero(o_gpu: torch.Tensor, row_mask_o: np.ndarray, what=""):
    """Rows that see no key hold +0.0 exactly (bf16 bit pattern 0)."""
    bits = o_gpu.contiguous().view(torch.int16).cpu().numpy()
    sel = bits[row_mask_o]
    assert np.all(sel == 0), f"{what}: fully masked rows are not +0.0"


def np64(t: torch.Tensor) -> np.ndarray:
    return t.double().numpy()
