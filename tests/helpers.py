"""Shared helpers of the GPU parity tests: oracle-side references and the tolerance rules.

Tolerances:
  * FP8 codes, scales and top-k indices: bit-exact.
  * logits: |I_gpu - I_ref| <= 1e-3 * |I_ref| + 1e-5 * M_ref, where M_ref = sum_h |w'| ReLU(...)
    is the magnitude of the summed terms (the sum cancels, so its rounding error scales with M, not
    with |I|: the fp32 accumulation of 128 exact FP8 products and the 64-term head sum each stay
    below ~2^-20 M, well inside 1e-5 M; 1e-3 |I| is the stated relative bar).
  * attention output: max |o_gpu - o_ref| <= 2e-2 on unit-variance data; lse within 1e-3.
"""
import numpy as np
import torch

import oracle

LOGIT_REL = 1e-3
LOGIT_MAG = 1e-5
ATTN_ABS = 2e-2
LSE_ABS = 1e-3
TOPK_GAP_REL = 1e-4


def bf16_to_np_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def oracle_pool(wl) -> np.ndarray:
    pool = np.zeros((wl.num_pages, oracle.PAGE_BYTES), np.uint8)
    bad = oracle.store_index_k(wl.index_keys(), wl.token_slots(), pool)
    assert bad == 0
    return pool


def check_logits(got_rows: np.ndarray, ref_rows: np.ndarray, mag_rows: np.ndarray, vis: np.ndarray):
    """got/ref/mag: [n, >= max vis]; only s < vis[i] is compared."""
    worst = 0.0
    for i, v in enumerate(vis):
        g = got_rows[i, :v].astype(np.float64)
        r = ref_rows[i, :v].astype(np.float64)
        m = mag_rows[i, :v]
        assert np.all(np.isfinite(g)), f"row {i}: non-finite logits"
        err = np.abs(g - r)
        bound = LOGIT_REL * np.abs(r) + LOGIT_MAG * m
        bad = err > bound
        assert not bad.any(), (f"row {i}: {bad.sum()} logits out of tolerance; worst at s={int(np.argmax(err - bound))} "
                               f"got {g[np.argmax(err - bound)]} ref {r[np.argmax(err - bound)]}")
        if v:
            worst = max(worst, float(np.max(err / np.maximum(bound, 1e-30))))
    return worst


def kth_gap_ok(ref_row: np.ndarray, k: int) -> bool:
    """True when the k-th and (k+1)-th largest reference logits are separated by more than the
    near-tie band, so the top-k set is unique under any admissible rounding."""
    if ref_row.shape[0] <= k:
        return True
    s = np.sort(ref_row.astype(np.float64))[::-1]
    a, b = s[k - 1], s[k]
    return (a - b) > TOPK_GAP_REL * max(abs(a), abs(b), 1e-30)


def check_topk_valid(idx_row: np.ndarray, ref_row: np.ndarray, k: int, mag_row=None):
    """A top-k row is valid when it has min(k, v) distinct in-range ascending indices, -1 after,
    and every kept logit is >= every dropped one up to the logit tolerance."""
    v = ref_row.shape[0]
    n = min(k, v)
    kept = idx_row[:n]
    assert np.all(idx_row[n:] == -1)
    assert np.all(kept >= 0) and np.all(kept < v)
    assert np.all(np.diff(kept) > 0)
    if n < v:
        mask = np.ones(v, bool)
        mask[kept] = False
        lo_kept = ref_row[kept].min()
        hi_drop = ref_row[mask].max()
        tol = LOGIT_REL * abs(hi_drop) + (LOGIT_MAG * float(mag_row.max()) if mag_row is not None else 0.0)
        assert lo_kept >= hi_drop - 2 * tol


def check_attention(out_gpu: np.ndarray, lse_gpu: np.ndarray, out_ref: np.ndarray, lse_ref: np.ndarray):
    err = np.abs(out_gpu - out_ref)
    assert err.max() <= ATTN_ABS, f"attention max abs err {err.max()}"
    fin = np.isfinite(lse_ref)
    assert np.array_equal(fin, np.isfinite(lse_gpu))
    if fin.any():
        assert np.abs(lse_gpu[fin] - lse_ref[fin]).max() <= LSE_ABS
    return float(err.max())
