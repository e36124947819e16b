"""Pins of the oracle's per-head projections around the absorbed attention (the absorbed latent
query and the value up-projection) and of its single-rounding float64 -> bf16 conversion: exact
rational rounding, integer brute force, identity weights, and the attention identities that make
the absorbed form equal to the unabsorbed one."""
import math
from fractions import Fraction

import numpy as np
import torch

import oracle


def bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_value(bits):
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def exact_bf16_round(q: Fraction) -> float:
    """Nearest bf16 of a rational (ties to even), by exhaustive comparison of the two neighbours."""
    if q == 0:
        return 0.0
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = math.floor(math.log2(a))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)                          # bf16 shares fp32's exponent range (subnormals below)
    ulp = Fraction(2) ** (e - 7)
    lo = (a // ulp) * ulp
    hi = lo + ulp
    if a - lo < hi - a:
        r = lo
    elif a - lo > hi - a:
        r = hi
    else:
        r = lo if (lo / ulp) % 2 == 0 else hi
    return sign * float(r)


def test_f64_to_bf16_is_one_correct_rounding():
    rng = np.random.default_rng(500)
    x = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-30, 30, 2000),
                        # values within one fp32 ulp of a bf16 midpoint, where two roundings fail
                        (1.0 + (2 * rng.integers(0, 128, 200) + 1) / 256.0) * (1 + rng.choice([-1, 1], 200) * 2.0 ** -30)])
    got = bf16_value(oracle.f64_to_bf16_array(x))
    for xi, gi in zip(x, got):
        assert gi == exact_bf16_round(Fraction(float(xi))), (xi, gi)


def test_absorb_integer_brute_force():
    rng = np.random.default_rng(501)
    T, N, P, L = 3, 2, 5, 7
    q = rng.integers(-4, 5, (T, N, P)).astype(np.float64)
    w = rng.integers(-4, 5, (N, P, L)).astype(np.float64)
    got = bf16_value(oracle.mla_absorb_q(bf16_bits(q), bf16_bits(w)))
    for t in range(T):
        for n in range(N):
            for l in range(L):
                assert got[t, n, l] == sum(int(q[t, n, p]) * int(w[n, p, l]) for p in range(P))


def test_v_up_integer_brute_force():
    rng = np.random.default_rng(502)
    T, N, L, V = 2, 3, 6, 4
    o = rng.integers(-4, 5, (T, N, L)).astype(np.float64)
    w = rng.integers(-4, 5, (N, L, V)).astype(np.float64)
    got = bf16_value(oracle.mla_v_up(bf16_bits(o), bf16_bits(w)))
    for t in range(T):
        for n in range(N):
            for v in range(V):
                assert got[t, n, v] == sum(int(o[t, n, l]) * int(w[n, l, v]) for l in range(L))


def test_absorb_rounds_the_exact_sum_once():
    rng = np.random.default_rng(503)
    T, N, P, L = 2, 2, 128, 16
    q = bf16_bits(rng.standard_normal((T, N, P)))
    w = bf16_bits(rng.standard_normal((N, P, L)) * 0.1)
    got = bf16_value(oracle.mla_absorb_q(q, w))
    qv, wv = bf16_value(q), bf16_value(w)
    for t in range(T):
        for n in range(N):
            for l in range(0, L, 5):
                exact = sum(Fraction(float(qv[t, n, p])) * Fraction(float(wv[n, p, l])) for p in range(P))
                assert got[t, n, l] == exact_bf16_round(exact)


def test_identity_weights_copy_the_query_and_heads_stay_apart():
    rng = np.random.default_rng(504)
    T, N = 4, 3
    q = bf16_bits(rng.standard_normal((T, N, 128)))
    w = np.zeros((N, 128, 512))
    w[0, :, :128] = np.eye(128)                   # head 0: copy into dims 0..127
    w[1, :, 384:] = 2.0 * np.eye(128)             # head 1: twice the query into dims 384..511
    got = bf16_value(oracle.mla_absorb_q(q, bf16_bits(w)))
    qv = bf16_value(q)
    assert np.array_equal(got[:, 0, :128], qv[:, 0]) and not got[:, 0, 128:].any()
    assert np.array_equal(got[:, 1, 384:], 2.0 * qv[:, 1]) and not got[:, 1, :384].any()
    assert not got[:, 2].any()                    # head 2's weights are zero


def test_absorbed_scores_equal_unabsorbed_scores():
    """q_nope . k_nope with k_nope = W_UK c (the unabsorbed key) equals the absorbed query
    ql = q_nope W_UK_T dotted with the latent row c (integer data: every step exact)."""
    rng = np.random.default_rng(505)
    T, N, P, L = 2, 4, 128, 512
    w_uk = rng.integers(-2, 3, (L, N, P)).astype(np.float64)      # kv_b_proj's qk_nope part (L, N, P)
    w_uk_t = np.transpose(w_uk, (1, 2, 0))                         # (N, P, L)
    q = rng.integers(-2, 3, (T, N, P)).astype(np.float64)
    c = rng.integers(-2, 3, (5, L)).astype(np.float64)             # latent rows
    ql = bf16_value(oracle.mla_absorb_q(bf16_bits(q), bf16_bits(w_uk_t)))
    for n in range(N):
        k_nope = c @ w_uk[:, n, :]                                 # [5, P]
        for t in range(T):
            assert np.array_equal(ql[t, n] @ c.T, k_nope @ q[t, n])


def test_v_up_of_the_latent_output_is_the_unabsorbed_output():
    """sum_i p_i (c_i W_UV) == (sum_i p_i c_i) W_UV: the value up-projection of the latent
    attention output equals attention over the up-projected values, to bf16 rounding."""
    rng = np.random.default_rng(506)
    T, N, L, V, n_keys = 3, 4, 512, 128, 50
    w_uv = rng.standard_normal((N, L, V)) / math.sqrt(L)
    w_uv_b = bf16_value(bf16_bits(w_uv))
    c = bf16_value(bf16_bits(rng.standard_normal((n_keys, L))))
    p = rng.random((T, N, n_keys))
    p /= p.sum(-1, keepdims=True)
    o_lat = np.einsum("tnk,kl->tnl", p, c)
    o_lat_b = bf16_bits(o_lat)
    got = bf16_value(oracle.mla_v_up(o_lat_b, bf16_bits(w_uv)))
    unabsorbed = np.einsum("tnk,knv->tnv", p, np.einsum("kl,nlv->knv", c, w_uv_b))
    # the only differences: o_lat rounded to bf16 before the projection, the output rounded to bf16
    mag = np.einsum("tnl,nlv->tnv", np.abs(o_lat), np.abs(w_uv_b))
    assert np.all(np.abs(got - unabsorbed) <= 2.0 ** -8 * np.abs(unabsorbed) + 2.0 ** -8 * mag)
    assert np.abs(got - unabsorbed).max() > 0        # not trivially equal


def test_projection_magnitudes_bound_the_sums():
    rng = np.random.default_rng(507)
    q = bf16_bits(rng.standard_normal((2, 3, 128)))
    w = bf16_bits(rng.standard_normal((3, 128, 512)))
    out, mag = oracle.mla_absorb_q(q, w, want_mag=True)
    assert np.all(np.abs(bf16_value(out)) <= mag * (1 + 2.0 ** -8))
    o = bf16_bits(rng.standard_normal((2, 3, 512)))
    wv = bf16_bits(rng.standard_normal((3, 512, 128)))
    out2, mag2 = oracle.mla_v_up(o, wv, want_mag=True)
    assert np.all(np.abs(bf16_value(out2)) <= mag2 * (1 + 2.0 ** -8))
