"""Pins of the oracle's compressed-KV (DSV4, compress ratio 4) functions: the compressed visible
length in closed form, the indexer and top-k over compressed entries against the plain ones on
the visible prefix, and the window + compressed + sink attention against a numpy float64 brute
force, the sink's limits (no sink: the plain sparse attention; a dominant sink: zero output), a
single key in closed form and the empty case."""
import numpy as np
import pytest
import torch

import oracle

RATIO = 4


def _bf16(x):
    return torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _val(bits):
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).double().numpy()


def _case(seed, lens, q_len, window=16, k=8, H=4):
    rng = np.random.default_rng(seed)
    B = len(lens)
    cu_q = np.concatenate([[0], np.cumsum([q_len] * B)]).astype(np.int32)
    T = int(cu_q[-1])
    swa_pages_per = [(L + 63) // 64 for L in lens]
    cmp_pages_per = [((L // RATIO) + 63) // 64 + 1 for L in lens]
    swa_bt = np.full((B, max(swa_pages_per)), -1, np.int32)
    cmp_bt = np.full((B, max(cmp_pages_per)), -1, np.int32)
    perm = rng.permutation(sum(swa_pages_per) + 2)
    permc = rng.permutation(sum(cmp_pages_per) + 2)
    o = oc = 0
    for b in range(B):
        swa_bt[b, :swa_pages_per[b]] = perm[o:o + swa_pages_per[b]]
        cmp_bt[b, :cmp_pages_per[b]] = permc[oc:oc + cmp_pages_per[b]]
        o += swa_pages_per[b]
        oc += cmp_pages_per[b]
    swa = _bf16(rng.standard_normal((perm.size, 64, 576)) * 0.5)
    cmp = _bf16(rng.standard_normal((permc.size, 64, 576)) * 0.5)
    q = _bf16(rng.standard_normal((T, H, 576)) * 0.2)
    idx = np.full((T, k), -1, np.int32)
    for r in range(T):
        vc = oracle.visible_len_cmp(np.array(lens, np.int32), cu_q, r, RATIO)
        n = min(k - 2, vc)
        if n > 0:
            idx[r, :n] = rng.choice(vc, n, replace=False)
        idx[r, k - 1] = vc + 3            # past the visible compressed entries: skipped
    sinks = rng.standard_normal(H).astype(np.float32)
    return dict(q=q, swa=swa, cmp=cmp, swa_bt=swa_bt, cmp_bt=cmp_bt, seq_lens=np.array(lens, np.int32), cu_q=cu_q,
                idx=idx, sinks=sinks, window=window, T=T, H=H, scale=576 ** -0.5)


def test_visible_len_cmp_closed_form():
    lens = np.array([100, 7, 4096], np.int32)
    cu_q = np.array([0, 3, 4, 6], np.int32)
    for r in range(6):
        b = int(np.searchsorted(cu_q, r, side="right") - 1)
        p = lens[b] - (cu_q[b + 1] - cu_q[b]) + (r - cu_q[b])
        assert oracle.visible_len_cmp(lens, cu_q, r, RATIO) == (p + 1) // RATIO


def test_indexer_and_topk_over_compressed_entries_are_the_plain_ones_on_the_prefix():
    rng = np.random.default_rng(31)
    lens = [600, 129, 8]
    cu_q = np.array([0, 2, 3, 4], np.int32)
    T = 4
    n_cmp = [L // RATIO + 1 for L in lens]
    mp = max((n + 63) // 64 for n in n_cmp)
    bt = np.arange(len(lens) * mp, dtype=np.int32).reshape(len(lens), mp)
    pool = np.zeros((bt.size, oracle.PAGE_BYTES), np.uint8)
    for b, n in enumerate(n_cmp):
        keys = _bf16(rng.standard_normal((n, 128)))
        slots = bt[b, np.arange(n) // 64].astype(np.int64) * 64 + np.arange(n) % 64
        oracle.store_index_k(keys, slots, pool)
    q = _bf16(rng.standard_normal((T, 64, 128)))
    w = (rng.standard_normal((T, 64)) * 0.1).astype(np.float32)
    rows = np.arange(T)
    sl = np.array(lens, np.int32)
    lg4 = oracle.indexer_logits(q, w, pool, bt, sl, cu_q, rows, 200, cmp_ratio=RATIO)
    # on the visible compressed prefix the logits are the plain rule's over the same cache
    for r in rows:
        vc = oracle.visible_len_cmp(sl, cu_q, r, RATIO)
        assert np.all(np.isnan(lg4[r, vc:]))
        assert np.all(np.isfinite(lg4[r, :vc]))
        plain = oracle.indexer_logits(q, w, pool, bt, sl, cu_q, [r], 800)
        assert np.array_equal(lg4[r, :vc], plain[0, :vc])
    idx4 = oracle.topk(lg4, sl, cu_q, rows, 16, cmp_ratio=RATIO)
    for r in rows:
        vc = oracle.visible_len_cmp(sl, cu_q, r, RATIO)
        order = np.argsort(-lg4[r, :vc].astype(np.float64), kind="stable")[:min(16, vc)]
        want = np.full(16, -1, np.int32)
        want[:len(order)] = np.sort(order)
        assert np.array_equal(idx4[r], want)


def _brute(c, rows):
    """numpy float64: gather the window and the selected compressed rows, softmax with the sink."""
    H = c["H"]
    out = np.zeros((len(rows), H, 512))
    lse = np.zeros((len(rows), H))
    for i, r in enumerate(rows):
        b = int(np.searchsorted(c["cu_q"], r, side="right") - 1)
        q_len = c["cu_q"][b + 1] - c["cu_q"][b]
        v = c["seq_lens"][b] - q_len + (r - c["cu_q"][b]) + 1
        keys = []
        for pos in range(max(0, v - c["window"]), v):
            keys.append(_val(c["swa"][c["swa_bt"][b, pos // 64], pos % 64]))
        for e in c["idx"][r]:
            if 0 <= e < v // RATIO:
                keys.append(_val(c["cmp"][c["cmp_bt"][b, e // 64], e % 64]))
        K = np.array(keys).reshape(-1, 576)
        qv = _val(c["q"][r])                              # [H, 576]
        S = c["scale"] * qv @ K.T                         # [H, n]
        z = np.concatenate([S, c["sinks"].astype(np.float64)[:, None]], axis=1)
        m = z.max(1, keepdims=True)
        e = np.exp(z - m)
        D = e.sum(1)
        out[i] = (e[:, :-1] / D[:, None]) @ K[:, :512]
        lse[i] = m[:, 0] + np.log(D)
    return out, lse


def _run(c, rows, sinks=None):
    return oracle.dsv4_attention(c["q"], c["swa"], c["swa_bt"], c["cmp"], c["cmp_bt"], c["seq_lens"], c["cu_q"],
                                 c["idx"], c["window"], c["sinks"] if sinks is None else sinks, c["scale"], rows)


def test_dsv4_attention_matches_numpy_brute_force():
    c = _case(32, [300, 9, 70], 2)
    rows = np.arange(c["T"])
    out, lse, bad = _run(c, rows)
    assert bad == c["T"]                                   # the one past-the-end entry per row
    ref_o, ref_l = _brute(c, rows)
    assert np.allclose(out, ref_o, atol=1e-12, rtol=1e-10)
    assert np.allclose(lse, ref_l, atol=1e-12, rtol=1e-12)


def test_without_sink_it_is_the_sparse_attention_over_the_union():
    c = _case(33, [200, 130], 1, window=24, k=6)
    rows = np.arange(c["T"])
    out, lse, _ = _run(c, rows, sinks=np.full(c["H"], -np.inf, np.float32))
    # one pool holding both caches; each row's window positions and selected entries as indices
    swa_p, cmp_p = c["swa"].shape[0], c["cmp"].shape[0]
    pool = np.concatenate([c["swa"], c["cmp"]])
    B = len(c["seq_lens"])
    span = max(c["swa_bt"].shape[1], 1) * 64
    bt = np.full((B, c["swa_bt"].shape[1] + c["cmp_bt"].shape[1]), -1, np.int32)
    bt[:, :c["swa_bt"].shape[1]] = c["swa_bt"]
    bt[:, c["swa_bt"].shape[1]:] = np.where(c["cmp_bt"] >= 0, c["cmp_bt"] + swa_p, -1)
    kk = c["window"] + c["idx"].shape[1]
    idx = np.full((c["T"], kk), -1, np.int32)
    for r in rows:
        b = int(np.searchsorted(c["cu_q"], r, side="right") - 1)
        v = c["seq_lens"][b]
        win = np.arange(max(0, v - c["window"]), v)
        idx[r, :len(win)] = win
        sel = [e for e in c["idx"][r] if 0 <= e < v // RATIO]
        idx[r, c["window"]:c["window"] + len(sel)] = np.array(sel, np.int64) + span
    big = np.full(c["seq_lens"].shape, span + c["cmp_bt"].shape[1] * 64, np.int32)
    ref_o, ref_l = oracle.sparse_mla(c["q"], pool, bt, big, c["cu_q"], idx, c["scale"], rows)
    assert np.allclose(out, ref_o, atol=1e-12) and np.allclose(lse, ref_l, atol=1e-12)


def test_sink_limits_single_key_and_empty_rows():
    c = _case(34, [1, 5], 1, window=1, k=4)
    rows = np.arange(c["T"])
    c["idx"][:] = -1                                       # window only: one key per row
    out, lse, _ = _run(c, rows)
    for i, r in enumerate(rows):
        b = r
        v = c["seq_lens"][b]
        kv = _val(c["swa"][c["swa_bt"][b, (v - 1) // 64], (v - 1) % 64])
        for h in range(c["H"]):
            S = c["scale"] * _val(c["q"][r, h]) @ kv
            s = float(c["sinks"][h])
            w = 1.0 / (1.0 + np.exp(s - S))
            assert np.allclose(out[i, h], w * kv[:512], atol=1e-12)
            assert np.isclose(lse[i, h], np.logaddexp(S, s))
    out_big, lse_big, _ = _run(c, rows, sinks=np.full(c["H"], 80.0, np.float32))
    assert np.abs(out_big).max() < 1e-30 and np.allclose(lse_big, 80.0)
    c["window"] = 0
    out0, lse0, _ = _run(c, rows)
    assert not out0.any() and np.array_equal(lse0, np.tile(c["sinks"].astype(np.float64), (c["T"], 1)))
