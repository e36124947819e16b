"""CPU checks of the key-prologue parity bar (helpers.compare_prologue_pools): a pool written from
keys normalised in fp32 with another summation order (what a kernel may do) passes it, the oracle's
own pool passes it exactly, and a code moved two E4M3 steps, or a scale moved by 2^-4, fails it."""
import numpy as np
import pytest
import torch

import oracle
from helpers import compare_prologue_pools

DI = 128


def _bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _f32(bits):
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).float().numpy()


def _norm_fp32_tree(x_bits, w, b, eps):
    """LayerNorm in fp32 with a pairwise summation tree (a stand-in for a kernel's evaluation)."""
    x = _f32(x_bits).astype(np.float32)

    def tree(v):
        s = np.array([(v[4 * l] + v[4 * l + 1]) + (v[4 * l + 2] + v[4 * l + 3]) for l in range(32)], np.float32)
        m = 1
        while m < 32:
            for l in range(0, 32, 2 * m):
                s[l] = np.float32(s[l] + s[l + m])
            m *= 2
        return s[0]

    mean = np.float32(tree(x) * np.float32(1 / 128))
    d = (x - mean).astype(np.float32)
    var = np.float32(tree((d * d).astype(np.float32)) * np.float32(1 / 128))
    rstd = np.float32(1) / np.sqrt(np.float32(var + np.float32(eps)))
    return _bf16_bits(((d * rstd).astype(np.float32) * w + b).astype(np.float32))


def _store_plain(pre, slots, pool):
    """Quantise and store bf16 keys without the rotation (oracle steps), as the fused path does."""
    for t in range(pre.shape[0]):
        codes, sc = oracle.quant128(oracle.bf16_bits_to_f64(pre[t]).astype(np.float32))
        pg, row = int(slots[t]) >> 6, int(slots[t]) & 63
        pool[pg, row * 128:row * 128 + 128] = codes
        pool[pg, 8192 + 4 * row:8192 + 4 * row + 4] = np.frombuffer(np.float32(sc).tobytes(), np.uint8)


def _case(seed=7, n=2000, pages=40, rotate=True):
    rng = np.random.default_rng(seed)
    keys = _bf16_bits(rng.standard_normal((n, DI)) * rng.uniform(0.01, 30.0, (n, 1)) + rng.standard_normal((n, 1)))
    w = rng.standard_normal(DI).astype(np.float32)
    b = rng.standard_normal(DI).astype(np.float32)
    max_pos = 1024
    f = 10000.0 ** (-np.arange(0, 64, 2, dtype=np.float64) / 64.0)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * f[None, :]
    cs = np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)
    pos = rng.integers(0, max_pos, n).astype(np.int64)
    slots = rng.permutation(pages * 64)[:n].astype(np.int64)
    ref = np.zeros((pages, oracle.PAGE_BYTES), np.uint8)
    assert oracle.store_index_k_prologue(keys, w, b, 1e-6, cs, pos, slots, ref, rotate=rotate) == 0
    # the "kernel": fp32 norm, then the oracle's rope and store
    pre = np.stack([oracle.rope64(_norm_fp32_tree(keys[t], w, b, 1e-6), cs[pos[t]]) for t in range(n)])
    alt = np.zeros_like(ref)
    if rotate:
        assert oracle.store_index_k(pre, slots, alt) == 0
    else:
        _store_plain(pre, slots, alt)
    return keys, w, b, cs, pos, slots, ref, alt


def test_bar_accepts_the_oracle_itself_exactly():
    keys, w, b, cs, pos, slots, ref, _ = _case(n=300, pages=8)
    assert compare_prologue_pools(ref, ref, keys, w, b, 1e-6, cs, pos, slots, False, True, True, False,
                                  key="bar_selfcheck") == (300, 0)


@pytest.mark.parametrize("rotate", [True, False])
def test_bar_accepts_an_fp32_norm_with_another_summation_order(rotate):
    keys, w, b, cs, pos, slots, ref, alt = _case(n=3000, pages=60, rotate=rotate)
    # with the rotation, a moved norm output reaches every code of the token, so some codes move;
    # without it, a one-unit move of a norm output rarely crosses an E4M3 rounding boundary
    assert rotate == (not np.array_equal(alt, ref))
    n_exact, n_boundary = compare_prologue_pools(alt, ref, keys, w, b, 1e-6, cs, pos, slots, False, True, rotate,
                                                 False, key="bar_selfcheck")
    assert n_boundary >= int(rotate) and n_exact + n_boundary == len(slots)


@pytest.mark.parametrize("what", ["code", "scale"])
def test_bar_rejects_a_code_two_steps_off_or_a_moved_scale(what):
    keys, w, b, cs, pos, slots, ref, _ = _case(n=300, pages=8)
    bad = ref.copy()
    t = 17
    pg, row = int(slots[t]) >> 6, int(slots[t]) & 63
    if what == "code":
        d = int(np.argmax(bad[pg, row * 128:row * 128 + 128] & 0x7F))   # the largest code: E4M3 steps of 16 or 32
        c = int(bad[pg, row * 128 + d])
        bad[pg, row * 128 + d] = (c & 0x80) | ((c & 0x7F) - 2)
    else:
        s = np.frombuffer(bad[pg, 8192 + 4 * row:8192 + 4 * row + 4].tobytes(), np.float32)[0] * np.float32(1.25)
        bad[pg, 8192 + 4 * row:8192 + 4 * row + 4] = np.frombuffer(np.float32(s).tobytes(), np.uint8)
    with pytest.raises(AssertionError):
        compare_prologue_pools(bad, ref, keys, w, b, 1e-6, cs, pos, slots, False, True, True, False,
                               key="bar_selfcheck")
