"""Pins of the oracle's indexer logits (brute force with torch/numpy, closed forms, causal rule) and
of its top-k (stable argsort prefix, brute force over all subsets)."""
import itertools

import numpy as np
import pytest
import torch

import oracle
from deepseek_sparse_attention_paged_gb300 import workloads


def e4m3_values(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_quant_rows(x_bf16):
    """Per-128 quantisation of bf16 rows with torch calls: returns (dequantised float64, scale)."""
    t = torch.from_numpy(np.ascontiguousarray(x_bf16).view(np.int16)).view(torch.bfloat16).to(torch.float32)
    amax = t.abs().amax(dim=-1, keepdim=True)
    s = torch.clamp(amax, min=torch.tensor(1e-4)) / torch.tensor(448.0)
    codes = (t / s).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return e4m3_values(codes), s.squeeze(-1).to(torch.float64).numpy()


def build_oracle_pool(wl):
    pool = np.zeros((wl.num_pages, oracle.PAGE_BYTES), np.uint8)
    assert oracle.store_index_k(wl.index_keys(), wl.token_slots(), pool) == 0
    return pool


def brute_force_logits(wl, pool, r):
    """I[r, s] for s < v_r, written independently with numpy einsum and torch's FP8 decode."""
    cu = wl.cu_q
    b = int(np.searchsorted(cu, r, side="right") - 1)
    v = int(wl.visible_lens()[r])
    qdq, qs = torch_quant_rows(wl.index_q()[r])                  # [64,128], [64]
    wq = wl.weights()[r].astype(np.float64) * qs
    s = np.arange(v)
    pages = wl.block_table[b, s // 64]
    codes = pool[pages][:, :8192].reshape(-1, 64, 128)[np.arange(v), s % 64]
    scales = pool[pages][:, 8192:].copy().view(np.float32).reshape(-1, 64)[np.arange(v), s % 64]
    kdq = e4m3_values(codes)                                     # [v,128]
    dots = kdq @ qdq.T                                           # [v,64]
    return (np.maximum(dots * scales[:, None].astype(np.float64), 0.0) * wq[None, :]).sum(1)


def test_logits_match_brute_force_tiny():
    wl = workloads.make("tiny")
    pool = build_oracle_pool(wl)
    rows = np.arange(wl.T)
    ld = wl.max_seq_len
    got, mag, bad = oracle.indexer_logits(wl.index_q(), wl.weights(), pool, wl.block_table, wl.seq_lens,
                                          wl.cu_q, rows, ld, want_mag=True)
    assert bad == 0
    for r in rows:
        v = int(wl.visible_lens()[r])
        ref = brute_force_logits(wl, pool, r)
        assert np.all(np.abs(got[r, :v].astype(np.float64) - ref) <= 2.0 ** -23 * mag[r, :v] + 1e-30)
        assert np.all(np.isnan(got[r, v:]))   # nothing past the visible length is written


def test_logits_closed_form_single_head():
    # hand-built one-page pool: key 0 = 0.5 * e_0 exactly, key 1 = -0.5 * e_0
    pool = np.zeros((1, oracle.PAGE_BYTES), np.uint8)
    pool[0, 0] = 0x38            # 1.0
    pool[0, 128] = 0xB8          # -1.0
    pool[0, 8192:8200] = np.array([0.5, 0.5], np.float32).view(np.uint8)
    q = np.zeros((1, 64, 128), np.uint16)
    q[0, 7, 0] = 0x4000          # bf16 2.0 in head 7 only
    w = np.zeros((1, 64), np.float32)
    w[0, 7] = 1.0
    bt = np.array([[0]], np.int32)
    out = oracle.indexer_logits(q, w, pool, bt, np.array([2], np.int32), np.array([0, 1], np.int32),
                                np.array([0]), 2)
    # ReLU(q . k): +1.0 for key 0, ReLU(-1.0) = 0 for key 1, up to the fp32 query scale
    assert abs(out[0, 0] - 1.0) < 1e-6
    assert out[0, 1] == 0.0


def test_logits_causal_rows_next_n():
    wl = workloads.make_custom("mtp_small", 5, [130, 70], 2, topk=64, heads=16)
    pool = build_oracle_pool(wl)
    vis = wl.visible_lens()
    assert vis.tolist() == [129, 130, 69, 70]
    out = oracle.indexer_logits(wl.index_q(), wl.weights(), pool, wl.block_table, wl.seq_lens, wl.cu_q,
                                np.arange(4), 130)
    for r in range(4):
        assert np.all(np.isfinite(out[r, :vis[r]])) and np.all(np.isnan(out[r, vis[r]:]))
        ref = brute_force_logits(wl, pool, r)
        assert np.allclose(out[r, :vis[r]], ref, rtol=1e-5, atol=1e-7)


def test_logits_rotate_q_flag_equals_prerotated_q():
    wl = workloads.make("tiny")
    pool = build_oracle_pool(wl)
    q = wl.index_q()
    qrot = np.stack([np.stack([oracle.rotate128(q[r, h]) for h in range(64)]) for r in range(wl.T)])
    a = oracle.indexer_logits(q, wl.weights(), pool, wl.block_table, wl.seq_lens, wl.cu_q, np.arange(2),
                              1000, rotate_q=True)
    b = oracle.indexer_logits(qrot, wl.weights(), pool, wl.block_table, wl.seq_lens, wl.cu_q, np.arange(2),
                              1000)
    assert np.array_equal(a, b, equal_nan=True)


# ------------------------------------------------------------------ top-k

def topk_one(x, k):
    lg = np.asarray(x, np.float32)[None, :]
    n = lg.shape[1]
    return oracle.topk(lg, np.array([n], np.int32), np.array([0, 1], np.int32), np.array([0]), k)[0]


def test_topk_equals_stable_argsort_prefix():
    rng = np.random.default_rng(31)
    for n, k in ((1000, 256), (5000, 2048), (300, 299), (64, 1)):
        x = rng.integers(-20, 20, n).astype(np.float32)      # many ties
        x[rng.integers(0, n, 5)] = -0.0
        order = np.argsort(-x, kind="stable")[:k]
        ref = np.sort(order)
        got = topk_one(x, k)
        assert np.array_equal(got[:len(ref)], ref)
        assert np.all(got[len(ref):] == -1)


def test_topk_short_rows_keep_all():
    x = np.random.default_rng(32).standard_normal(100).astype(np.float32)
    got = topk_one(x, 256)
    assert np.array_equal(got[:100], np.arange(100)) and np.all(got[100:] == -1)


def test_topk_signed_zero_and_nan():
    x = np.array([-0.0, 0.0, np.nan, -1.0, 0.0, -0.0], np.float32)
    assert topk_one(x, 3).tolist() == [0, 1, 4]          # +-0 tie, lower indices win
    assert topk_one(x, 5).tolist() == [0, 1, 3, 4, 5]    # NaN is never preferred


def test_topk_brute_force_all_subsets():
    rng = np.random.default_rng(33)
    for _ in range(60):
        n = int(rng.integers(1, 11))
        k = int(rng.integers(1, n + 1))
        x = rng.integers(-3, 3, n).astype(np.float32)
        winners = []
        for sub in itertools.combinations(range(n), k):
            inside = set(sub)
            ok = all((x[i] > x[j]) or (x[i] == x[j] and i < j)
                     for i in inside for j in range(n) if j not in inside)
            if ok:
                winners.append(sub)
        assert len(winners) == 1
        assert topk_one(x, k).tolist() == list(winners[0])


def test_topk_uses_visible_length_per_row():
    # two rows of one request with next_n = 2: row 0 sees 5 keys, row 1 sees 6
    lg = np.array([[0, 1, 2, 3, 4, 99, 7], [0, 1, 2, 3, 4, 99, 7]], np.float32)
    idx = oracle.topk(lg, np.array([6], np.int32), np.array([0, 2], np.int32), np.array([0, 1]), 2)
    assert idx.tolist() == [[3, 4], [4, 5]]


def _forced_brute(row, k, n_init, n_local):
    """Forced positions first (they count as +inf, lower index first among equals), then the
    largest of the rest by (value descending, index ascending); the kept indices ascending."""
    v = len(row)
    forced = sorted(set(range(min(n_init, v))) | set(range(max(0, v - n_local), v)))
    val = [np.inf if i in forced else float(row[i]) for i in range(v)]
    order = sorted(range(v), key=lambda i: (-val[i] if not np.isnan(val[i]) else np.inf, i))
    kept = sorted(order[:min(k, v)])
    return kept + [-1] * (k - len(kept))


@pytest.mark.parametrize("v,k,n_init,n_local", [(50, 8, 2, 3), (50, 4, 3, 3), (10, 20, 2, 2), (200, 16, 0, 5),
                                                 (200, 16, 5, 0), (30, 10, 40, 0), (30, 10, 0, 40)])
def test_topk_forced_matches_brute_force(v, k, n_init, n_local):
    rng = np.random.default_rng(900 + v + k + n_init)
    row = rng.standard_normal(v).astype(np.float32)
    row[v // 2] = np.inf                      # a real +inf competes with the forced ones by index
    got = oracle.topk_forced(row[None, :], np.array([v], np.int32), np.array([0, 1], np.int32), [0], k,
                             n_init, n_local)[0]
    assert list(got) == _forced_brute(row, k, n_init, n_local)


def test_topk_forced_keeps_every_forced_position_that_fits():
    rng = np.random.default_rng(910)
    v, k = 1000, 64
    row = rng.standard_normal(v).astype(np.float32) + 100.0   # every real logit large
    got = oracle.topk_forced(row[None, :], np.array([v], np.int32), np.array([0, 1], np.int32), [0], k, 4, 16)[0]
    assert set(range(4)) <= set(got) and set(range(v - 16, v)) <= set(got)
    plain = oracle.topk(row[None, :], np.array([v], np.int32), np.array([0, 1], np.int32), [0], k)[0]
    assert set(got) - set(range(4)) - set(range(v - 16, v)) <= set(plain)
