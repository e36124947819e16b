"""Pins of the oracle's absorbed sparse MLA: dense equivalence, an independent numpy softmax,
absorbed == unabsorbed with random projection weights, weight sums, single-token and permutation
invariants, skipping of padding / out-of-range entries, and the log-sum-exp merge."""
import math

import numpy as np
import pytest
import torch

import oracle
from deepseek_sparse_attention_paged_gb300 import workloads


def bf16_value(bits):
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def small_wl(seed=41, lens=(150, 90), heads=16, q_len=1):
    return workloads.make_custom("mla_small", seed, list(lens), q_len, topk=64, heads=heads)


def gather_rows(wl, b, positions):
    pages = wl.block_table[b, np.asarray(positions) // 64]
    return bf16_value(wl.latent_pool()[pages, np.asarray(positions) % 64])   # [n,576]


def numpy_attention(q, C, scale):
    S = scale * (C @ q)
    m = S.max()
    p = np.exp(S - m)
    l = p.sum()
    return (p / l) @ C[:, :512], m + math.log(l)


def test_dense_matches_numpy_softmax():
    wl = small_wl()
    out, lse = oracle.dense_mla(wl.mla_q(), wl.latent_pool(), wl.block_table, wl.seq_lens, wl.cu_q,
                                wl.scale, np.arange(wl.T))
    q = bf16_value(wl.mla_q())
    for r in range(wl.T):
        C = gather_rows(wl, r, np.arange(wl.seq_lens[r]))
        for h in range(wl.heads):
            o, l = numpy_attention(q[r, h], C, wl.scale)
            assert np.allclose(out[r, h], o, rtol=1e-10, atol=1e-12)
            assert abs(lse[r, h] - l) < 1e-10


def test_sparse_with_all_positions_equals_dense():
    wl = small_wl()
    k = 160
    idx = np.full((wl.T, k), -1, np.int32)
    rng = np.random.default_rng(42)
    for r in range(wl.T):
        v = wl.seq_lens[r]
        idx[r, :v] = rng.permutation(v)
    s_out, s_lse = oracle.sparse_mla(wl.mla_q(), wl.latent_pool(), wl.block_table, wl.seq_lens, wl.cu_q,
                                     idx, wl.scale, np.arange(wl.T))
    d_out, d_lse = oracle.dense_mla(wl.mla_q(), wl.latent_pool(), wl.block_table, wl.seq_lens, wl.cu_q,
                                    wl.scale, np.arange(wl.T))
    assert np.allclose(s_out, d_out, rtol=1e-12, atol=1e-13)
    assert np.allclose(s_lse, d_lse, rtol=1e-12, atol=1e-13)


def test_absorbed_equals_unabsorbed():
    """Unabsorbed MLA (k_nope = W_UK c, v = W_UV^T c, 192-wide score q_nope.k_nope + q_pe.k_pe)
    against the oracle's absorbed form (latent query ql = q_nope W_UK, 576-wide score on the
    latent rows), with v_up (W_UV) applied to the absorbed latent output.  Integer-valued q_nope,
    W_UK and dyadic q_pe make the absorbed query exactly representable in bf16, so the two forms
    must agree to double rounding."""
    rng = np.random.default_rng(43)
    wl = small_wl(heads=4)
    H = wl.heads
    W_UK = rng.choice([-1.0, 0.0, 1.0], size=(H, 128, 512), p=[1 / 64, 62 / 64, 1 / 64])
    W_UV = rng.standard_normal((H, 512, 128)) / math.sqrt(512)
    q_nope = rng.choice([-1.0, 0.0, 1.0], size=(wl.T, H, 128))
    q_pe = rng.integers(-16, 16, size=(wl.T, H, 64)) / 8.0
    ql = np.einsum("thp,hpl->thl", q_nope, W_UK)
    q_abs = np.concatenate([ql, q_pe], axis=-1)
    q_bits = bf16_bits(q_abs)
    assert np.array_equal(bf16_value(q_bits), q_abs)
    k = 200
    idx = np.full((wl.T, k), -1, np.int32)
    for r in range(wl.T):
        idx[r, :wl.seq_lens[r]] = np.arange(wl.seq_lens[r])
    out, lse = oracle.sparse_mla(q_bits, wl.latent_pool(), wl.block_table, wl.seq_lens, wl.cu_q, idx,
                                 wl.scale, np.arange(wl.T))
    for r in range(wl.T):
        C = gather_rows(wl, r, np.arange(wl.seq_lens[r]))
        for h in range(H):
            k_nope = C[:, :512] @ W_UK[h].T                        # [n,128]
            v = C[:, :512] @ W_UV[h]                               # [n,128]
            S = wl.scale * (k_nope @ q_nope[r, h] + C[:, 512:] @ q_pe[r, h])
            p = np.exp(S - S.max())
            lse_unabs = S.max() + math.log(p.sum())
            p /= p.sum()
            o_unabs = p @ v
            o_abs = out[r, h] @ W_UV[h]
            assert np.allclose(o_abs, o_unabs, rtol=1e-9, atol=1e-11)
            assert abs(lse[r, h] - lse_unabs) < 1e-9


def test_weights_sum_to_one_and_single_token():
    wl = small_wl()
    rng = np.random.default_rng(44)
    idx = np.full((wl.T, 64), -1, np.int32)
    for r in range(wl.T):
        idx[r, :40] = np.sort(rng.choice(wl.seq_lens[r], 40, replace=False))
    out, lse, psum, bad = oracle.sparse_mla(wl.mla_q(), wl.latent_pool(), wl.block_table, wl.seq_lens,
                                            wl.cu_q, idx, wl.scale, np.arange(wl.T), want_psum=True)
    assert bad == 0
    assert np.allclose(psum, 1.0, atol=1e-12)
    one = np.full((wl.T, 64), -1, np.int32)
    one[:, 5] = 17
    out1, lse1 = oracle.sparse_mla(wl.mla_q(), wl.latent_pool(), wl.block_table, wl.seq_lens, wl.cu_q,
                                   one, wl.scale, np.arange(wl.T))
    q = bf16_value(wl.mla_q())
    for r in range(wl.T):
        c = gather_rows(wl, r, [17])[0]
        assert np.array_equal(out1[r], np.broadcast_to(c[:512], out1[r].shape))
        assert np.allclose(lse1[r], wl.scale * (q[r] @ c), rtol=1e-12)


def test_permutation_invariance_and_skips():
    wl = small_wl()
    rng = np.random.default_rng(45)
    idx = np.full((wl.T, 64), -1, np.int32)
    for r in range(wl.T):
        idx[r, :50] = np.sort(rng.choice(wl.seq_lens[r], 50, replace=False))
    out, lse = oracle.sparse_mla(wl.mla_q(), wl.latent_pool(), wl.block_table, wl.seq_lens, wl.cu_q, idx,
                                 wl.scale, np.arange(wl.T))
    perm = np.stack([rng.permutation(row) for row in idx])
    out_p, lse_p = oracle.sparse_mla(wl.mla_q(), wl.latent_pool(), wl.block_table, wl.seq_lens, wl.cu_q,
                                     perm, wl.scale, np.arange(wl.T))
    assert np.allclose(out, out_p, rtol=1e-12, atol=1e-14) and np.allclose(lse, lse_p, rtol=1e-13)
    # entries past the visible length are skipped and counted, like -1 padding is skipped
    bad_idx = idx.copy()
    bad_idx[:, 60] = 100000
    out_b, lse_b, _, bad = oracle.sparse_mla(wl.mla_q(), wl.latent_pool(), wl.block_table, wl.seq_lens,
                                             wl.cu_q, bad_idx, wl.scale, np.arange(wl.T), want_psum=True)
    assert bad == wl.T and np.array_equal(out_b, out) and np.array_equal(lse_b, lse)


def test_empty_selection_gives_zero_and_neg_inf():
    wl = small_wl()
    idx = np.full((wl.T, 64), -1, np.int32)
    out, lse = oracle.sparse_mla(wl.mla_q(), wl.latent_pool(), wl.block_table, wl.seq_lens, wl.cu_q, idx,
                                 wl.scale, np.arange(wl.T))
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_lse_merge_of_halves_equals_whole():
    wl = small_wl()
    rng = np.random.default_rng(46)
    idx = np.full((wl.T, 64), -1, np.int32)
    for r in range(wl.T):
        idx[r, :64] = np.sort(rng.choice(wl.seq_lens[r], 64, replace=False))
    a, b = idx.copy(), idx.copy()
    a[:, 32:] = -1
    b[:, :32] = -1
    rows = np.arange(wl.T)
    args = (wl.mla_q(), wl.latent_pool(), wl.block_table, wl.seq_lens, wl.cu_q)
    o, l = oracle.sparse_mla(*args, idx, wl.scale, rows)
    oa, la = oracle.sparse_mla(*args, a, wl.scale, rows)
    ob, lb = oracle.sparse_mla(*args, b, wl.scale, rows)
    om, lm = oracle.lse_merge(oa, la, ob, lb)
    assert np.allclose(om, o, rtol=1e-12, atol=1e-14) and np.allclose(lm, l, rtol=1e-13)
    # merging with an empty part is the identity
    e = np.full_like(idx, -1)
    oe, le = oracle.sparse_mla(*args, e, wl.scale, rows)
    om2, lm2 = oracle.lse_merge(o, l, oe, le)
    assert np.allclose(om2, o, rtol=1e-15) and np.array_equal(lm2, l)
