"""GPU parity of the indexer prologue calls against the CPU oracle, through the C ABI:
dsa_store_index_k_prologue (key norm, rotary embedding, rotate, quantise, paged store) token by
token against the oracle's exact norm (codes and scale equal, or -- for the few tokens whose exact
norm output lies within the fp32 evaluation's error of a bf16 rounding boundary -- admissible by the
bar in helpers.prologue_token_admissible), and dsa_indexer_rope_q (rotary embedding of the indexer
query, the same fp32 operations on both sides) bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from deepseek_sparse_attention_paged_gb300 import capi
from helpers import compare_prologue_pools

pytestmark = pytest.mark.gpu


def _bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _cos_sin_cache(max_pos, base=10000.0):
    """Rotary table of a 64-dim rope head: row p = [cos(p f_i) for i < 32, sin(p f_i) for i < 32],
    f_i = base^(-2i / 64)."""
    f = base ** (-np.arange(0, 64, 2, dtype=np.float64) / 64.0)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * f[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def _keys(rng, n):
    x = rng.standard_normal((n, 128)) * rng.uniform(0.01, 30.0, (n, 1)) + rng.standard_normal((n, 1))
    x[5] = 2.5                                # constant key: LayerNorm output is the bias
    x[6] = 0.0                                # zero key
    return _bf16_bits(x)


@pytest.mark.parametrize("rms,interleaved,rotate,ue8m0", [(r, i, o, False) for r in (False, True)
                                                          for i in (False, True) for o in (True, False)] +
                         [(False, False, True, True), (True, True, False, True)])
def test_store_prologue_matches_oracle(rms, interleaved, rotate, ue8m0):
    rng = np.random.default_rng(300 + 8 * ue8m0 + 4 * rotate + 2 * rms + interleaved)
    n, pages, max_pos = 1500, 30, 4096
    keys = _keys(rng, n)
    w = rng.standard_normal(128).astype(np.float32)
    b = rng.standard_normal(128).astype(np.float32)
    eps = 1e-6
    cs = _cos_sin_cache(max_pos)
    pos = rng.integers(0, max_pos, n).astype(np.int64)
    slots = rng.permutation(pages * 64)[:n].astype(np.int64)
    slots[10] = -1                            # padding token
    pos[11] = max_pos                         # position out of range
    pos[12] = -3
    slots[13] = pages * 64 + 7                # slot past the pool
    flags = ((capi.DSA_NORM_RMS if rms else 0) | (capi.DSA_ROPE_INTERLEAVED if interleaved else 0) |
             (0 if rotate else capi.DSA_K_NO_ROTATE) | (capi.DSA_SCALE_UE8M0 if ue8m0 else 0))

    ref = np.full((pages, oracle.PAGE_BYTES), 0x33, np.uint8)
    bad = oracle.store_index_k_prologue(keys, w, None if rms else b, eps, cs, pos, slots, ref, rms=rms,
                                        neox=not interleaved, rotate=rotate, ue8m0=ue8m0)
    assert bad == 3
    pool = torch.full((pages, oracle.PAGE_BYTES), 0x33, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    capi.dsa_store_index_k_prologue(_bf16_dev(keys), torch.from_numpy(w).cuda(),
                                    None if rms else torch.from_numpy(b).cuda(), eps, torch.from_numpy(cs).cuda(),
                                    torch.from_numpy(pos).cuda(), torch.from_numpy(slots).cuda(), pool,
                                    flags=flags, dev_err=err)
    got = pool.cpu().numpy()
    compare_prologue_pools(got, ref, keys, w, None if rms else b, eps, cs, pos, slots, rms, not interleaved, rotate,
                           ue8m0)
    st, word = capi.dsa_read_device_error(err)
    assert st == capi.DSA_ERR_DEVICE_BOUNDS
    assert word == capi.DSA_DEVERR_POSITION | capi.DSA_DEVERR_SLOT_RANGE


def test_store_prologue_equals_norm_rope_then_store():
    """The fused call stores what the plain store writes for the oracle's normed, rotated keys
    (up to the norm's rounding-boundary tokens, under the same bar)."""
    rng = np.random.default_rng(310)
    n, pages, max_pos = 300, 8, 1000
    keys = _keys(rng, n)
    w = rng.uniform(0.5, 1.5, 128).astype(np.float32)
    b = (rng.standard_normal(128) * 0.1).astype(np.float32)
    cs = _cos_sin_cache(max_pos)
    pos = rng.integers(0, max_pos, n).astype(np.int64)
    slots = rng.permutation(pages * 64)[:n].astype(np.int64)
    pre = np.stack([oracle.rope64(oracle.k_norm128(keys[t], w, b, 1e-5), cs[pos[t]]) for t in range(n)])
    plain = torch.zeros((pages, oracle.PAGE_BYTES), dtype=torch.uint8, device="cuda")
    capi.dsa_store_index_k(_bf16_dev(pre), torch.from_numpy(slots).cuda(), plain)
    fused = torch.zeros_like(plain)
    capi.dsa_store_index_k_prologue(_bf16_dev(keys), torch.from_numpy(w).cuda(), torch.from_numpy(b).cuda(), 1e-5,
                                    torch.from_numpy(cs).cuda(), torch.from_numpy(pos).cuda(),
                                    torch.from_numpy(slots).cuda(), fused)
    compare_prologue_pools(fused.cpu().numpy(), plain.cpu().numpy(), keys, w, b, 1e-5, cs, pos, slots, False, True,
                           True, False, key="key_prologue_vs_store")


def test_store_prologue_empty_and_bad_flags():
    pool = torch.zeros((1, oracle.PAGE_BYTES), dtype=torch.uint8, device="cuda")
    w = torch.ones(128, device="cuda")
    b = torch.zeros(128, device="cuda")
    cs = torch.from_numpy(_cos_sin_cache(4)).cuda()
    e64 = torch.zeros(0, dtype=torch.int64, device="cuda")
    capi.dsa_store_index_k_prologue(torch.zeros((0, 128), dtype=torch.bfloat16, device="cuda"), w, b, 1e-6, cs,
                                    e64, e64, pool)
    torch.cuda.synchronize()
    assert int(pool.sum()) == 0
    one = torch.zeros(1, dtype=torch.int64, device="cuda")
    with pytest.raises(capi.DSAError):
        capi.dsa_store_index_k_prologue(torch.zeros((1, 128), dtype=torch.bfloat16, device="cuda"), w, b, 1e-6, cs,
                                        one, one, pool, flags=0x40)


@pytest.mark.parametrize("interleaved", [False, True])
@pytest.mark.parametrize("T", [37, 1300])   # one head per warp / 16 heads per warp
def test_rope_q_bit_exact_and_in_place(interleaved, T):
    rng = np.random.default_rng(320 + interleaved + T)
    max_pos = 70000
    q = _bf16_bits(rng.standard_normal((T, 64, 128)) * rng.uniform(0.1, 10.0, (T, 64, 1)))
    cs = _cos_sin_cache(max_pos)
    pos = rng.integers(0, max_pos, T).astype(np.int64)
    pos[3] = max_pos                          # out of range: row copied
    pos[4] = max_pos - 1
    ref, bad = oracle.rope_q(q, cs, pos, neox=not interleaved)
    assert bad == 1
    flags = capi.DSA_ROPE_INTERLEAVED if interleaved else 0
    qd = _bf16_dev(q)
    csd = torch.from_numpy(cs).cuda()
    pd = torch.from_numpy(pos).cuda()
    out = torch.empty_like(qd)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    capi.dsa_indexer_rope_q(qd, csd, pd, out, flags=flags, dev_err=err)
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, ref)
    assert capi.dsa_read_device_error(err) == (capi.DSA_ERR_DEVICE_BOUNDS, capi.DSA_DEVERR_POSITION)
    capi.dsa_indexer_rope_q(qd, csd, pd, qd, flags=flags)          # in place
    assert np.array_equal(qd.view(torch.int16).cpu().numpy().view(np.uint16), ref)


def test_rope_q_then_rotated_logits_match_oracle_chain():
    """Query rope feeding the logits call (with the Hadamard query prologue) gives the oracle's
    logits of the oracle-roped query."""
    from deepseek_sparse_attention_paged_gb300 import workloads
    from deepseek_sparse_attention_paged_gb300.pipeline import DeviceBatch
    from helpers import check_logits, oracle_pool

    wl = workloads.make("tiny")
    db = DeviceBatch(wl, with_latent=False)
    rng = np.random.default_rng(330)
    max_pos = 4096
    cs = _cos_sin_cache(max_pos)
    pos = rng.integers(0, max_pos, wl.T).astype(np.int64)
    q_raw = wl.index_q()
    q_rope, bad = oracle.rope_q(q_raw, cs, pos)
    assert bad == 0
    qd = _bf16_dev(q_raw)
    capi.dsa_indexer_rope_q(qd, torch.from_numpy(cs).cuda(), torch.from_numpy(pos).cuda(), qd)
    lg = torch.full((wl.T, db.ld), float("nan"), dtype=torch.float32, device="cuda")
    db.indexer_logits(q=qd, logits=lg, flags=capi.DSA_Q_ROTATE)
    rows = np.arange(wl.T)
    ref, mag, bad = oracle.indexer_logits(q_rope, wl.weights(), oracle_pool(wl), wl.block_table, wl.seq_lens,
                                          wl.cu_q, rows, db.ld, rotate_q=True, want_mag=True)
    assert bad == 0
    check_logits(lg.cpu().numpy(), ref, mag, wl.visible_lens())
