"""Pins of the oracle's Hadamard rotation, per-128 FP8 quantisation and paged index-K store.

The Hadamard matrix is built here independently, by the Sylvester recursion and by its closed
form H[i, j] = (-1)^popcount(i & j); the quantisation is re-derived with torch library calls."""
import math

import numpy as np
import pytest
import torch

import oracle

N = 128


def sylvester(n):
    h = np.array([[1]], np.int64)
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def closed_form_hadamard(n):
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    pc = np.vectorize(lambda v: bin(int(v)).count("1"))(i & j)
    return np.where(pc % 2 == 0, 1, -1).astype(np.int64)


def bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_value(bits):
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()


def test_hadamard_matrix_invariant():
    H = sylvester(N)
    assert np.array_equal(H, closed_form_hadamard(N))
    assert np.array_equal(H @ H.T, N * np.eye(N, dtype=np.int64))


def test_fwht_basis_vectors_give_hadamard_rows():
    H = sylvester(N)
    for i in range(N):
        e = np.zeros(N, np.float32)
        e[i] = 1.0
        assert np.array_equal(oracle.fwht128(e), H[:, i].astype(np.float32))


def test_fwht_equals_matrix_product_on_integers():
    rng = np.random.default_rng(21)
    H = sylvester(N)
    for _ in range(50):
        x = rng.integers(-1000, 1000, N)
        assert np.array_equal(oracle.fwht128(x.astype(np.float32)).astype(np.int64), H @ x)


def test_fwht_fp32_error_bound_on_reals():
    rng = np.random.default_rng(22)
    H = sylvester(N).astype(np.float64)
    for _ in range(50):
        x = rng.standard_normal(N).astype(np.float32)
        exact = H @ x.astype(np.float64)
        got = oracle.fwht128(x).astype(np.float64)
        # 7 butterfly levels, each rounding once relative to at most sum |x|
        assert np.max(np.abs(got - exact)) <= 7 * 2.0 ** -24 * np.abs(x).sum() * 2


def test_rotation_exact_inputs_match_torch_pipeline():
    # small integers: every fp32 butterfly is exact, so the rotation is
    # bf16(fp32(H x) * fp32(1/sqrt(128))) computed here with torch
    rng = np.random.default_rng(23)
    H = sylvester(N)
    c = np.float32(1.0 / math.sqrt(N))
    for _ in range(50):
        xi = rng.integers(-100, 100, N)
        xb = bf16_bits(xi.astype(np.float32))
        assert np.array_equal(bf16_value(xb), xi.astype(np.float32))
        hx = (H @ xi).astype(np.float32)
        expect = bf16_bits(hx * c)
        assert np.array_equal(oracle.rotate128(xb), expect)


def test_rotation_preserves_norm_to_bf16_rounding():
    rng = np.random.default_rng(24)
    for _ in range(50):
        xb = bf16_bits(rng.standard_normal(N).astype(np.float32))
        x = bf16_value(xb).astype(np.float64)
        y = bf16_value(oracle.rotate128(xb)).astype(np.float64)
        assert abs(np.linalg.norm(y) - np.linalg.norm(x)) <= 2.0 ** -8 * np.linalg.norm(x)
        # rotation is its own inverse up to rounding: H/sqrt(n) is symmetric orthogonal
        back = sylvester(N) @ y / math.sqrt(N)
        assert np.max(np.abs(back - x)) <= 2.0 ** -7 * np.max(np.abs(x)) * 4


def torch_quant(y):
    t = torch.from_numpy(np.asarray(y, np.float32))
    amax = t.abs().max()
    s = torch.clamp(amax, min=torch.tensor(1e-4, dtype=torch.float32)) / torch.tensor(448.0)
    q = (t / s)
    codes = q.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return codes, np.float32(s.item())


def test_quant_matches_torch_pipeline():
    rng = np.random.default_rng(25)
    for scale in (1.0, 1e-3, 37.0):
        for _ in range(40):
            y = (rng.standard_normal(N) * scale).astype(np.float32)
            codes, s = oracle.quant128(y)
            tc, ts = torch_quant(y)
            assert s == ts
            assert np.array_equal(codes, tc)


def test_quant_amax_maps_to_448_and_error_bound():
    rng = np.random.default_rng(26)
    grid = np.sort(np.unique(np.abs(
        torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy())))
    for _ in range(40):
        y = rng.standard_normal(N).astype(np.float32)
        codes, s = oracle.quant128(y)
        i = int(np.argmax(np.abs(y)))
        assert codes[i] & 0x7F == 0x7E
        dec = np.array([oracle.e4m3_decode(int(c)) for c in codes])
        t = np.abs(y.astype(np.float64) / np.float64(s))
        # half the gap between the two grid points around |y/s|
        k = np.clip(np.searchsorted(grid, t), 1, len(grid) - 1)
        half_gap = (grid[k] - grid[k - 1]) / 2
        assert np.all(np.abs(np.abs(dec) - t) <= half_gap * (1 + 1e-6))


def test_quant_zero_vector():
    codes, s = oracle.quant128(np.zeros(N, np.float32))
    assert np.all(codes == 0)
    assert s == np.float32(np.float32(1e-4) / np.float32(448.0))


def test_store_layout_and_padding_slots():
    rng = np.random.default_rng(27)
    pages = 3
    pool = np.full((pages, oracle.PAGE_BYTES), 0xAB, np.uint8)
    keys = bf16_bits(rng.integers(-50, 50, (4, N)).astype(np.float32))
    slots = np.array([5, -1, 2 * 64 + 63, 3 * 64], np.int64)  # last one is past the pool
    bad = oracle.store_index_k(keys, slots, pool)
    assert bad == 1
    H = sylvester(N)
    c = np.float32(1.0 / math.sqrt(N))
    touched = np.zeros_like(pool, bool)
    for t, slot in ((0, 5), (2, 2 * 64 + 63)):
        page, row = divmod(slot, 64)
        xi = bf16_value(keys[t]).astype(np.int64)
        y = bf16_value(bf16_bits((H @ xi).astype(np.float32) * c))
        codes, s = torch_quant(y)
        assert np.array_equal(pool[page, row * 128:(row + 1) * 128], codes)
        assert pool[page, 8192 + row * 4:8192 + row * 4 + 4].view(np.float32)[0] == s
        touched[page, row * 128:(row + 1) * 128] = True
        touched[page, 8192 + row * 4:8192 + row * 4 + 4] = True
    assert np.all(pool[~touched] == 0xAB)


def test_ue8m0_scale_is_the_smallest_power_of_two_not_below_the_plain_scale():
    rng = np.random.default_rng(77)
    cases = [rng.standard_normal(128) * 10.0 ** rng.uniform(-6, 3) for _ in range(200)]
    cases.append(np.full(128, 448.0 * 2.0 ** -3))        # plain scale exactly 2^-3: kept
    cases.append(np.zeros(128))                            # floor 1e-4 / 448
    for y in cases:
        y = np.asarray(y, np.float32)
        _, s_plain = oracle.quant128(y)
        codes, s = oracle.quant128(y, ue8m0=True)
        m, e = math.frexp(float(s))
        assert m == 0.5                                    # a power of two
        assert s >= s_plain and (s == s_plain or s / 2 < s_plain)
        # dividing by a power of two is exact: the codes are torch's conversion of y / s
        ref = torch.from_numpy(y / np.float32(s)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(codes, ref)
        dec = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        assert np.all(np.abs(dec) <= 448.0)


def test_ue8m0_key_store_writes_power_of_two_scales():
    """With ue8m0 the stored scale of every key (through the fused key prologue) is a power of two."""
    rng = np.random.default_rng(78)
    n, pages, max_pos = 64, 1, 128
    k_raw = bf16_bits(rng.standard_normal((n, 128)))
    w = np.ones(128, np.float32)
    b = np.zeros(128, np.float32)
    cs = np.concatenate([np.ones((max_pos, 32)), np.zeros((max_pos, 32))], axis=1).astype(np.float32)  # identity rope
    pos = np.arange(n, dtype=np.int64)
    slots = np.arange(n, dtype=np.int64)
    pool = np.zeros((pages, oracle.PAGE_BYTES), np.uint8)
    assert oracle.store_index_k_prologue(k_raw, w, b, 1e-6, cs, pos, slots, pool, ue8m0=True) == 0
    scales = pool[0, 64 * 128:].view(np.float32)
    for sc in scales:
        assert math.frexp(float(sc))[0] == 0.5


def test_ue8m0_query_equals_plain_when_the_plain_scale_is_a_power_of_two():
    """Query heads whose amax is 448 * 2^-j have a plain fp32 scale of exactly 2^-j, so the ue8m0
    and plain query quantisations coincide and so do the logits; for general heads they differ
    by no more than the FP8 rounding allows."""
    from deepseek_sparse_attention_paged_gb300 import workloads
    wl = workloads.make("tiny")
    pool = np.zeros((wl.num_pages, oracle.PAGE_BYTES), np.uint8)
    assert oracle.store_index_k(wl.index_keys(), wl.token_slots(), pool) == 0
    rng = np.random.default_rng(79)
    q = rng.standard_normal((wl.T, 64, 128)).astype(np.float32)
    q /= np.abs(q).max(axis=-1, keepdims=True)
    q *= (448.0 * 2.0 ** -rng.integers(2, 9, (wl.T, 64, 1))).astype(np.float32)
    qb = bf16_bits(q)
    assert np.all(bf16_value(qb).reshape(wl.T, 64, 128).__abs__().max(-1) == np.abs(q).max(-1))
    rows = np.arange(wl.T)
    plain = oracle.indexer_logits(qb, wl.weights(), pool, wl.block_table, wl.seq_lens, wl.cu_q, rows, 1000)
    pow2 = oracle.indexer_logits(qb, wl.weights(), pool, wl.block_table, wl.seq_lens, wl.cu_q, rows, 1000,
                                 ue8m0_q=True)
    assert np.array_equal(plain, pow2, equal_nan=True)
    qg = bf16_bits(rng.standard_normal((wl.T, 64, 128)) * 3.0)
    p2, mag, _ = oracle.indexer_logits(qg, wl.weights(), pool, wl.block_table, wl.seq_lens, wl.cu_q, rows, 1000,
                                       ue8m0_q=True, want_mag=True)
    pl = oracle.indexer_logits(qg, wl.weights(), pool, wl.block_table, wl.seq_lens, wl.cu_q, rows, 1000)
    v = wl.visible_lens()
    for i in range(wl.T):
        d = np.abs(p2[i, :v[i]].astype(np.float64) - pl[i, :v[i]])
        assert np.all(d <= 2.0 ** -3 * mag[i, :v[i]] + 1e-6)      # two e4m3 roundings of each product term
        assert d.max() > 0                                           # the formats do differ
