"""Pins of the oracle's FP8 latent-cache path (per-tensor FP8 quantisation of the latent cache and
of the decode query, sparse MLA over the FP8 cache) against torch's E4M3 conversion, exact
identities with the bf16 sparse MLA, and a numpy brute force."""
import numpy as np
import torch

import oracle

DQK, DV = 576, 512


def _bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _f32(bits):
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).float().numpy()


def _e4m3_values():
    return torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)


def test_quant_equals_torch_e4m3_of_the_fp32_quotient():
    rng = np.random.default_rng(40)
    x = _bf16_bits(rng.standard_normal(20000) * 3.0)
    for scale in (1.0, 0.0123, 3.7):
        got = oracle.quant_fp8_tensor(x, scale)
        q = (torch.from_numpy(_f32(x)) / torch.tensor(scale, dtype=torch.float32))   # one fp32 division
        inside = q.abs() <= 448.0
        ref = q.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(got[inside.numpy()], ref[inside.numpy()])
        # beyond the largest finite magnitude: saturated to +-448 (codes 0x7e / 0xfe)
        out = ~inside.numpy()
        assert np.all((got[out] & 0x7F) == 0x7E)


def test_store_layout_padding_and_range():
    rng = np.random.default_rng(41)
    n, pages = 50, 3
    lat = _bf16_bits(rng.standard_normal((n, DQK)))
    slots = rng.permutation(pages * 64)[:n].astype(np.int64)
    slots[4] = -1
    slots[7] = pages * 64 + 3        # past the pool
    pool = np.full((pages, 64, DQK), 0x5A, np.uint8)
    assert oracle.store_latent_fp8(lat, slots, 0.02, pool) == 1
    for t in range(n):
        if t in (4, 7):
            continue
        s = int(slots[t])
        assert np.array_equal(pool[s >> 6, s & 63], oracle.quant_fp8_tensor(lat[t], 0.02))
    written = {int(s) for t, s in enumerate(slots) if t not in (4, 7)}
    untouched = [s for s in range(pages * 64) if s not in written]
    assert all(np.all(pool[s >> 6, s & 63] == 0x5A) for s in untouched)


def _mla_case(seed, lens, heads, k):
    from deepseek_sparse_attention_paged_gb300 import workloads
    wl = workloads.make_custom("fp8_pin", seed, lens, 1, topk=k, heads=heads)
    rng = np.random.default_rng(seed)
    idx = np.full((wl.T, k), -1, np.int32)
    for r, v in enumerate(wl.visible_lens()):
        m = min(k, int(v))
        idx[r, :m] = np.sort(rng.choice(int(v), m, replace=False))
    return wl, idx


def test_fp8_mla_equals_bf16_mla_on_exactly_representable_values():
    """Queries and cache rows that are E4M3 values times power-of-two scales quantise exactly, so
    the FP8 path computes the bf16 path's definition on the same numbers: bit-identical results."""
    wl, idx = _mla_case(42, [300, 129], 16, 128)
    rng = np.random.default_rng(42)
    vals = _e4m3_values()
    finite = vals[np.isfinite(vals) & (np.abs(vals) <= 64)]
    k_scale, q_scale = 2.0 ** -5, 2.0 ** -3
    kv_vals = rng.choice(finite, (wl.num_pages, 64, DQK)) * k_scale
    q_vals = rng.choice(finite, (wl.T, wl.heads, DQK)) * q_scale
    kv_bf16, q_bf16 = _bf16_bits(kv_vals), _bf16_bits(q_vals)
    assert np.array_equal(_f32(kv_bf16), kv_vals.astype(np.float32))   # exact in bf16
    kv_fp8 = oracle.quant_fp8_tensor(kv_bf16, k_scale)
    rows = np.arange(wl.T)
    o8, l8 = oracle.sparse_mla_fp8(q_bf16, q_scale, kv_fp8, k_scale, wl.block_table, wl.seq_lens, wl.cu_q, idx,
                                   wl.scale, rows)
    o16, l16 = oracle.sparse_mla(q_bf16, kv_bf16, wl.block_table, wl.seq_lens, wl.cu_q, idx, wl.scale, rows)
    assert np.array_equal(o8, o16) and np.array_equal(l8, l16)


def test_fp8_mla_matches_numpy_brute_force():
    """Random (not representable) inputs: numpy dequantises torch's E4M3 codes of x / scale and runs
    the softmax attention in float64."""
    wl, idx = _mla_case(43, [200], 16, 64)
    rng = np.random.default_rng(43)
    kv_bf16 = _bf16_bits(rng.standard_normal((wl.num_pages, 64, DQK)))
    q_bf16 = _bf16_bits(rng.standard_normal((wl.T, wl.heads, DQK)))
    k_scale, q_scale = 0.011, 0.017
    kv_fp8 = oracle.quant_fp8_tensor(kv_bf16, k_scale)
    o, l = oracle.sparse_mla_fp8(q_bf16, q_scale, kv_fp8, k_scale, wl.block_table, wl.seq_lens, wl.cu_q, idx, wl.scale,
                                 np.arange(wl.T))
    vals = _e4m3_values()
    deq_kv = vals[kv_fp8] * np.float64(np.float32(k_scale))
    qq = (torch.from_numpy(_f32(q_bf16)) / torch.tensor(q_scale, dtype=torch.float32)).clamp(-448, 448)
    deq_q = vals[qq.to(torch.float8_e4m3fn).view(torch.uint8).numpy()] * np.float64(np.float32(q_scale))
    r = 0
    sel = idx[r][idx[r] >= 0]
    g = wl.block_table[0][sel >> 6].astype(np.int64) * 64 + (sel & 63)
    rowsv = deq_kv.reshape(-1, DQK)[g]
    for h in range(wl.heads):
        s = wl.scale * rowsv @ deq_q[r, h]
        p = np.exp(s - s.max())
        ref_o = (p / p.sum()) @ rowsv[:, :DV]
        assert np.allclose(o[r, h], ref_o, rtol=0, atol=1e-12)
        assert abs(l[r, h] - (s.max() + np.log(p.sum()))) <= 1e-12
