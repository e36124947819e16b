"""Pins of the oracle's int8 ("c8") indexer functions against what the pages and the mathematics fix:
numpy's IEEE fp16 conversion, the Hadamard matrix's closed form (one-hot columns, H H = 128 I),
properties of round-to-nearest-even quantisation, the page layout decoded independently, a numpy
brute force of the logits, and the unquantised score within the quantisation error bound."""
import numpy as np
import pytest
import scipy.linalg
import torch

import oracle

C = 181.0 / 2048.0          # bf16(128^-0.5): 0.08837890625


def _bf16(x):
    return torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_val(bits):
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).float().numpy()


# ------------------------------------------------------------------ fp16


def test_f16_decode_every_pattern_matches_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_decode(int(b)) for b in bits])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(got[~both_nan], ref[~both_nan])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_f32_to_f16_matches_numpy_rounding():
    rng = np.random.default_rng(11)
    vals = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * np.float32(10.0) ** rng.integers(-9, 6, 4000).astype(np.float32),
        np.float32(2.0) ** np.arange(-30, 17, dtype=np.float32),
        np.array([65504, 65519, 65520, 65536, 1e-8, 2.98e-8, 5.96e-8, 6.1e-5, -0.0, 0.0, np.inf, -np.inf],
                 np.float32),
    ])
    # exact halfway points between neighbouring fp16 values (ties go to the even mantissa)
    h = np.arange(0x0001, 0x7bff, 37, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    vals = np.concatenate([vals, ((lo + hi) / 2).astype(np.float32), -((lo + hi) / 2).astype(np.float32)])
    got = np.array([oracle.f32_to_f16(float(v)) for v in vals], np.uint16)
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------ rotation


def test_c8_rotation_of_one_hot_vectors_is_a_signed_hadamard_column():
    H = scipy.linalg.hadamard(128)
    for j in (0, 1, 5, 64, 127):
        for mag in (1.0, 2.0 ** -20, 3.0):
            x = np.zeros(128, np.float32)
            x[j] = mag
            y = _bf16_val(oracle.c8_rotate128(_bf16(x))).astype(np.float64)
            # the exact column entries +-c * mag, rounded once to bf16 (exact for powers of two)
            assert np.array_equal(y, _bf16_val(_bf16(H[j] * C * mag)).astype(np.float64))
            if mag != 3.0:
                assert np.array_equal(y, H[j] * C * mag)


def test_c8_rotation_of_two_spikes_adds_columns():
    H = scipy.linalg.hadamard(128)
    x = np.zeros(128, np.float32)
    x[3], x[100] = 1.0, -1.0
    y = _bf16_val(oracle.c8_rotate128(_bf16(x))).astype(np.float64)
    assert np.array_equal(y, (H[3] - H[100]) * C)


def test_c8_rotation_applied_twice_scales_by_128_c_squared():
    rng = np.random.default_rng(12)
    for _ in range(20):
        x = _bf16_val(_bf16(rng.standard_normal(128))).astype(np.float64)
        y = oracle.c8_rotate128(oracle.c8_rotate128(_bf16(x)))
        got = _bf16_val(y).astype(np.float64)
        want = x * 128 * C * C                     # H H = 128 I, every entry scaled by c
        # two bf16 roundings of the intermediate (each at most 2^-9 relative of its entries)
        bound = 2.0 ** -8 * np.abs(x).max() * 1.2 + 2.0 ** -9 * np.abs(want)
        assert np.all(np.abs(got - want) <= bound)


def test_c8_rotation_is_the_correctly_rounded_matrix_product():
    rng = np.random.default_rng(13)
    H = scipy.linalg.hadamard(128).astype(np.float64) * C
    for _ in range(10):
        xb = _bf16(rng.standard_normal(128) * 5)
        exact = _bf16_val(xb).astype(np.float64) @ H
        got = _bf16_val(oracle.c8_rotate128(xb)).astype(np.float64)
        # correctly rounded: within half a bf16 ulp of the exact product
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(exact), 1e-30))) - 7)
        assert np.all(np.abs(got - exact) <= ulp / 2 + 1e-300)


# ------------------------------------------------------------------ dynamic int8 quantisation


def test_quant_int8_ties_round_to_even_and_max_maps_to_127():
    y = np.zeros(128, np.float32)
    y[0] = 127.0                                    # scale exactly 1
    y[1:9] = [2.5, 3.5, -2.5, -3.5, 0.5, 1.5, 126.5, -0.5]
    codes, sc = oracle.quant_int8(y)
    assert sc == 1.0
    assert codes[0] == 127
    assert list(codes[1:9]) == [2, 4, -2, -4, 0, 2, 126, 0]


def test_quant_int8_properties():
    rng = np.random.default_rng(14)
    for t in range(50):
        y = (rng.standard_normal(128) * 10.0 ** rng.uniform(-6, 3)).astype(np.float32)
        codes, sc = oracle.quant_int8(y)
        amax = np.abs(y).max()
        i = int(np.argmax(np.abs(y)))
        assert abs(int(codes[i])) == 127 and np.sign(codes[i]) == np.sign(y[i])
        assert np.all(np.abs(codes.astype(np.int32)) <= 127)
        assert abs(sc - amax / 127) <= 2 ** -23 * amax / 127
        err = np.abs(codes.astype(np.float64) * sc - y.astype(np.float64))
        assert np.all(err <= sc * (0.5 + 1e-5))
        neg, _ = oracle.quant_int8(-y)
        assert np.array_equal(neg, -codes)
        order = np.argsort(y, kind="stable")
        assert np.all(np.diff(codes[order].astype(np.int32)) >= 0)


def test_quant_int8_zero_vector():
    codes, sc = oracle.quant_int8(np.zeros(128, np.float32))
    assert sc == 0.0 and not codes.any()


# ------------------------------------------------------------------ store


def test_store_c8_layout_padding_and_range():
    rng = np.random.default_rng(15)
    n, pages = 300, 8
    keys = _bf16(rng.standard_normal((n, 128)) * rng.uniform(0.01, 5, (n, 1)))
    slots = rng.permutation(pages * 64)[:n].astype(np.int64)
    slots[7] = -1
    slots[8] = pages * 64 + 1
    pool = np.full((pages, oracle.C8_PAGE_BYTES), 0xA5, np.uint8)
    assert oracle.store_index_k_c8(keys, slots, pool) == 1
    written = np.zeros((pages, 64), bool)
    for t in range(n):
        s = int(slots[t])
        if s < 0 or s >= pages * 64:
            continue
        pg, o = divmod(s, 64)
        written[pg, o] = True
        codes = pool[pg, o * 128:(o + 1) * 128].view(np.int8)
        sc16 = pool[pg, 8192 + 2 * o:8192 + 2 * o + 2].view(np.float16)[0]
        y = _bf16_val(oracle.c8_rotate128(keys[t]))
        want_codes, want_sc = oracle.quant_int8(y)
        assert np.array_equal(codes, want_codes)
        assert sc16 == np.float16(want_sc)
    for pg in range(pages):
        for o in range(64):
            if not written[pg, o]:
                assert np.all(pool[pg, o * 128:(o + 1) * 128] == 0xA5)
                assert np.all(pool[pg, 8192 + 2 * o:8192 + 2 * o + 2] == 0xA5)


# ------------------------------------------------------------------ logits


def _c8_case(seed, lens, q_per_req):
    rng = np.random.default_rng(seed)
    B = len(lens)
    cu_q = np.concatenate([[0], np.cumsum(q_per_req)]).astype(np.int32)
    T = int(cu_q[-1])
    max_pages = (max(lens) + 63) // 64
    num_pages = B * max_pages + 3
    perm = rng.permutation(num_pages)[: B * max_pages].astype(np.int32)
    bt = perm.reshape(B, max_pages)
    pool = np.zeros((num_pages, oracle.C8_PAGE_BYTES), np.uint8)
    kraw = []
    for b, L in enumerate(lens):
        k = _bf16(rng.standard_normal((L, 128)))
        slots = (bt[b, np.arange(L) // 64].astype(np.int64) * 64 + np.arange(L) % 64)
        oracle.store_index_k_c8(k, slots, pool)
        kraw.append(k)
    q = _bf16(rng.standard_normal((T, 64, 128)))
    w = (rng.standard_normal((T, 64)) * 0.05).astype(np.float32)
    return dict(q=q, w=w, pool=pool, bt=bt, seq_lens=np.array(lens, np.int32), cu_q=cu_q, T=T, kraw=kraw)


def test_logits_c8_match_a_numpy_brute_force():
    c = _c8_case(16, [70, 200, 1], [1, 3, 1])
    ld = 256
    rows = np.arange(c["T"])
    got, bad = oracle.indexer_logits_c8(c["q"], c["w"], c["pool"], c["bt"], c["seq_lens"], c["cu_q"], rows, ld)
    assert bad == 0
    pool = c["pool"]
    for r in rows:
        b = int(np.searchsorted(c["cu_q"], r, side="right") - 1)
        q_len = c["cu_q"][b + 1] - c["cu_q"][b]
        v = c["seq_lens"][b] - q_len + (r - c["cu_q"][b]) + 1
        cq = np.empty((64, 128), np.int64)
        qs = np.empty(64)
        for h in range(64):
            codes, sc = oracle.quant_int8(_bf16_val(oracle.c8_rotate128(c["q"][r, h])))
            cq[h] = codes
            qs[h] = float(np.float16(sc))
        w16 = c["w"][r].astype(np.float16).astype(np.float64)
        s = np.arange(v)
        pages = c["bt"][b, s // 64]
        ck = np.stack([pool[p, (t % 64) * 128:(t % 64 + 1) * 128].view(np.int8) for p, t in zip(pages, s)]).astype(np.int64)
        ks = np.array([pool[p, 8192 + 2 * (t % 64):8194 + 2 * (t % 64)].view(np.float16)[0] for p, t in zip(pages, s)],
                      np.float64)
        dots = ck @ cq.T                                               # [v, 64] exact integers
        ref = (np.maximum(dots * qs[None, :] * ks[:, None], 0.0) * w16[None, :]).sum(1).astype(np.float32)
        assert np.allclose(got[r, :v], ref, rtol=2e-7, atol=1e-30)
        assert np.all(np.isnan(got[r, v:]))


def test_logits_c8_close_to_the_unquantised_score():
    """int8 quantisation of both sides changes each head's dot product by at most
    |q|_1 dk + |k|_1 dq + 128 dq dk (dq, dk half the scales); the fp16 scales and weights add a
    relative 2^-11 each."""
    c = _c8_case(17, [150], [2])
    H = scipy.linalg.hadamard(128).astype(np.float64) * C
    rows = np.arange(c["T"])
    got, _ = oracle.indexer_logits_c8(c["q"], c["w"], c["pool"], c["bt"], c["seq_lens"], c["cu_q"], rows, 160)
    keys = _bf16_val(c["kraw"][0]).astype(np.float64)
    kr = np.stack([_bf16_val(oracle.c8_rotate128(_bf16(k))).astype(np.float64) for k in keys])
    k_sc = np.abs(kr).max(1) / 127
    for r in rows:
        v = 150 - 2 + r + 1
        qr = np.stack([_bf16_val(oracle.c8_rotate128(c["q"][r, h])).astype(np.float64) for h in range(64)])
        q_sc = np.abs(qr).max(1) / 127
        w = c["w"][r].astype(np.float64)
        dots = kr[:v] @ qr.T
        exact = (np.maximum(dots, 0) * w[None, :]).sum(1)
        ddot = (np.abs(qr).sum(1)[None, :] * k_sc[:v, None] / 2 + np.abs(kr[:v]).sum(1)[:, None] * q_sc[None, :] / 2
                + 128 * q_sc[None, :] * k_sc[:v, None] / 4)
        bound = (np.abs(w)[None, :] * (ddot + 4 * 2.0 ** -11 * np.abs(dots))).sum(1) * 1.01 + 1e-6
        assert np.all(np.abs(got[r, :v] - exact) <= bound)
        # and the quantised score is a real approximation (not trivially within a loose bound)
        assert np.corrcoef(got[r, :v], exact)[0, 1] > 0.999


def test_logits_c8_bad_page_is_counted_and_skipped():
    c = _c8_case(18, [130], [1])
    bt = c["bt"].copy()
    bt[0, 1] = c["pool"].shape[0] + 7
    got, bad = oracle.indexer_logits_c8(c["q"], c["w"], c["pool"], bt, c["seq_lens"], c["cu_q"], [0], 140)
    assert bad == 64
    assert np.all(np.isnan(got[0, 64:128])) and np.all(np.isfinite(got[0, :64]))
